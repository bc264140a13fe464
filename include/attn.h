/*
 * attn.h - C ABI of the GB300 (sm_103a) exact IO-aware attention library.
 *
 * The library computes exact multi-head scaled-dot-product attention and its
 * backward pass tile by tile, never writing an N x N score or probability
 * matrix to device memory.  What is computed, per batch b and head h, with
 * tau = `scale`:
 *
 *   S = tau Q K^T,  s_ij = -inf for j > i when `causal`,
 *   P = row softmax(S),  O = P V,  lse_i = ln sum_j exp(s_ij)
 *     (sj-techlog "FlashAttention 원 논문 해부", section "원 논문의 정의";
 *      wonbeomjang.kr FlashAttention-2 review, "개선 2: m과 l 대신 L만 저장")
 *
 *   dP = dO V^T,  D_i = sum_j P_ij dP_ij,  dS_ij = P_ij (dP_ij - D_i),
 *   dV = P^T dO,  dQ = tau dS K,  dK = tau dS^T Q
 *     (FlashAttention-2 review, sections "Backward Pass"; the factor tau
 *      comes from S = tau Q K^T).
 *
 * Conventions shared by every entry point
 *  - Layout: Q, K, V, O, dO, dQ, dK, dV are contiguous [B, H, N, d] arrays of
 *    16-bit floats (bfloat16 for the plain names, IEEE half for the `_f16`
 *    twins).  lse and D are contiguous [B, H, N] fp32.  dq_accum is a
 *    contiguous [B, H, N, d] fp32 workspace.
 *  - All pointers are DEVICE pointers of the current CUDA device and must be
 *    16-byte aligned.  The caller allocates and owns every buffer; the library
 *    allocates no device memory and keeps no per-call state.
 *  - Sizes: B, H, N >= 1; d is 64 or 128; B*H <= 2^31-1; B*H*N*d < 2^62;
 *    N <= 2^24 - 256.  scale must be finite and > 0 (callers usually pass
 *    1/sqrt(d)).
 *  - Causal masking is top-left aligned: key j is visible to query i iff
 *    j <= i.  Every query row therefore sees at least key 0.
 *  - Every call enqueues its kernels on `stream` (a cudaStream_t; NULL = the
 *    legacy default stream) and returns without synchronising.  Argument
 *    errors are detected on the host before anything is enqueued.  A launch
 *    failure returns ATTN_ERR_LAUNCH.  Kernels never trap: a bounded wait that
 *    runs out (about 2 s of unsuccessful barrier polls; the bound counts
 *    polls, so time the kernel spends preempted does not count) records
 *    ATTN_ERR_TIMEOUT in the library's device status word, read with
 *    attn_get_device_status().
 *  - Return value: an attn_status code (0 = success).  Nothing throws.
 *  - Per device, the first call looks up the device addresses of the
 *    library's status word (and, for attn_bwd_noalloc, of its workspace
 *    array) and keeps them for the life of the process.  Resetting a device
 *    (cudaDeviceReset) invalidates those addresses: do not call the library
 *    on a device after resetting it in the same process.
 */
#ifndef IO_AWARE_EXACT_GB300_ATTN_H
#define IO_AWARE_EXACT_GB300_ATTN_H

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_INVALID_ARG = 1,          /* null pointer, bad size, bad scale */
    ATTN_ERR_UNSUPPORTED_HEAD_DIM = 2, /* d not in {64, 128} */
    ATTN_ERR_MISALIGNED = 3,           /* a pointer is not 16-byte aligned */
    ATTN_ERR_UNSUPPORTED_DEVICE = 4,   /* current device is not sm_103 */
    ATTN_ERR_LAUNCH = 5,               /* CUDA launch / driver error */
    ATTN_ERR_TIMEOUT = 6,              /* a kernel's bounded wait ran out */
    ATTN_ERR_DEVICE_FAULT = 7,         /* CUDA reported an error while syncing */
    ATTN_ERR_SCRATCH_TOO_SMALL = 8     /* problem too large for attn_bwd_noalloc */
} attn_status;

/*
 * Forward pass.  Reads q, k, v [B,H,N,d]; writes o [B,H,N,d] and lse [B,H,N]
 * (natural-log logsumexp of each row's scaled, masked scores).  The row
 * statistics and output follow the FlashAttention-2 forward (FlashAttention-2
 * review, "결과: FlashAttention-2 Forward 알고리즘"): online softmax over key
 * blocks with one final division by the normaliser.
 */
int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
             int B, int H, int N, int d, int causal, float scale, void* stream);
int attn_fwd_f16(const void* q, const void* k, const void* v, void* o, float* lse,
                 int B, int H, int N, int d, int causal, float scale, void* stream);

/*
 * Forward pass for training: as attn_fwd, and additionally writes o32
 * [B,H,N,d] fp32, the same O before its rounding to 16 bits, for
 * attn_bwd_preprocess_o32 (the backward saves O, sj-techlog page, backward
 * section; here at accumulation precision).  Here each output row (o32 and
 * o) is normalised by the sum of the probabilities as rounded for the P V
 * product, so its weights sum to exactly 1; attn_fwd normalises by the exact
 * fp32 sum, so the two 16-bit outputs may differ in the last bit.  lse uses
 * the exact fp32 sum in both.  o32 must be non-NULL and 16-byte aligned.
 */
int attn_fwd_train(const void* q, const void* k, const void* v, void* o, float* o32, float* lse,
                   int B, int H, int N, int d, int causal, float scale, void* stream);
int attn_fwd_train_f16(const void* q, const void* k, const void* v, void* o, float* o32,
                       float* lse, int B, int H, int N, int d, int causal, float scale,
                       void* stream);

/*
 * Backward pre-processing.  Computes the softmax-gradient row term
 *   D_i = sum_j P_ij dP_ij,   P_ij = exp(s_ij - lse_i),   dP = dO V^T
 * (wonbeomjang.kr FlashAttention-2 review, "Backward Pass": D_i is the sum
 * over row i of P o dP, computed once ahead of the main loop) in fp32 from P
 * recomputed tile by tile and dP on the tensor cores, writes it to D [B,H,N],
 * and sets dq_accum [B,H,N,d] to zero.  Reads q, k, v, dO [B,H,N,d] and lse
 * [B,H,N] (from attn_fwd with the same q, k, v, causal, scale).  Must precede
 * attn_bwd on the same stream.
 *
 * The review also gives D_i = rowsum(dO_i o O_i); it is equal in exact
 * arithmetic, but O exists only rounded to 16 bits, and on rows whose
 * softmax is nearly one-hot dS = P (dP - D) cancels so that this rounding
 * alone exceeds the library's gradient tolerance.  Evaluating the definition
 * with the same fp32 P that attn_bwd uses avoids it, for the price of one
 * extra pass over S and dP.
 */
int attn_bwd_preprocess(const void* q, const void* k, const void* v, const void* dO,
                        const float* lse, float* D, float* dq_accum,
                        int B, int H, int N, int d, int causal, float scale, void* stream);
int attn_bwd_preprocess_f16(const void* q, const void* k, const void* v, const void* dO,
                            const float* lse, float* D, float* dq_accum,
                            int B, int H, int N, int d, int causal, float scale, void* stream);

/*
 * Backward pre-processing from the forward's fp32 O (the FlashAttention-2
 * review's D_i = rowsum(dO_i o O_i), "Backward Pass" of FlashAttention-2):
 * reads o32 [B,H,N,d] fp32 (from attn_fwd_train) and dO [B,H,N,d] 16-bit,
 * writes D [B,H,N] and zeroes dq_accum.  A memory-bound pass; gives the same
 * D as attn_bwd_preprocess to within the output tolerance, including on
 * nearly one-hot rows, because o32's weights sum to exactly 1.  Must precede
 * attn_bwd on the same stream.
 */
int attn_bwd_preprocess_o32(const float* o32, const void* dO, float* D, float* dq_accum,
                            int B, int H, int N, int d, void* stream);
int attn_bwd_preprocess_o32_f16(const float* o32, const void* dO, float* D, float* dq_accum,
                                int B, int H, int N, int d, void* stream);

/*
 * Backward pass (recomputation of S and P from lse, sj-techlog page, section
 * "forward가 끝난 뒤 backward는 무엇을 저장하고 무엇을 다시 계산하는가";
 * K/V-block outer loop of the FlashAttention-2 backward).  Reads q, k, v, dO
 * [B,H,N,d], lse and D [B,H,N] (from attn_fwd and attn_bwd_preprocess with
 * the same arguments), accumulates dS K into dq_accum (zeroed by the
 * preprocess) with fp32 atomics, and writes dq, dk, dv [B,H,N,d].
 * dq_accum is left holding dQ / scale.
 */
int attn_bwd(const void* q, const void* k, const void* v, const void* dO,
             const float* lse, const float* D, float* dq_accum,
             void* dq, void* dk, void* dv,
             int B, int H, int N, int d, int causal, float scale, void* stream);
int attn_bwd_f16(const void* q, const void* k, const void* v, const void* dO,
                 const float* lse, const float* D, float* dq_accum,
                 void* dq, void* dk, void* dv,
                 int B, int H, int N, int d, int causal, float scale, void* stream);

/*
 * Backward pass without caller-provided workspace (bf16).  The paper has no
 * counterpart: this entry point exists for callers that cannot allocate
 * device memory at the time of the call, for example plug-ins whose host
 * framework owns all allocations, or real-time programs that allocate
 * nothing after start-up.
 *
 * Computes exactly what attn_bwd_preprocess followed by attn_bwd compute,
 * reading q, k, v, dO [B,H,N,d] and lse [B,H,N] and writing dq, dk, dv
 * [B,H,N,d], but keeps D and the fp32 dQ accumulator in a fixed 16 MiB
 * device array that the library reserves on every GPU that loads it, until
 * the process exits.  It allocates nothing.
 *  - Size limit: ceil(B*H*N / 64) * 64 + B*H*N*d <= 4194304 (fp32 elements),
 *    e.g. B*H*N <= 32513 at d = 128 and <= 64527 at d = 64.  Larger problems
 *    return ATTN_ERR_SCRATCH_TOO_SMALL with nothing enqueued.
 *  - The first call on a device looks the array's device address up (once
 *    per device, with that device current).
 *  - The looked-up address is kept for the life of the process, so calling
 *    this entry point on a device after a cudaDeviceReset of that device is
 *    not supported (see the shared conventions above).
 *  - All calls on a device share the one array.  Each call overwrites D and
 *    zeroes the accumulator before use, so earlier contents do not matter,
 *    but calls whose kernels overlap on the GPU (different streams without
 *    ordering between them) race on the array and give wrong results.
 * Other conventions (alignment, errors, stream semantics) as for attn_bwd.
 */
int attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* dO,
                     const float* lse, void* dq, void* dk, void* dv,
                     int B, int H, int N, int d, int causal, float scale, void* stream);

/*
 * Grouped key / value heads (GQA; MQA when Hkv = 1).  The "v1에서 v3까지"
 * version table of the paldyn.com survey ("어텐션 비용 줄이기") lists GQA
 * support among FlashAttention-2's additions without defining it; the plain
 * reading taken here: q, dO, o, o32, dq are [B,H,N,d] and lse, D are [B,H,N]
 * as above, while k, v, dk, dv are [B,Hkv,N,d], and query head h reads K / V
 * head h / (H / Hkv) of the same batch entry (contiguous groups of H / Hkv
 * query heads share one K / V head).  dK and dV of a K / V head are the sums
 * over its group's query heads.  H must be a multiple of Hkv (>= 1), else
 * ATTN_ERR_INVALID_ARG with nothing enqueued.  With Hkv = H each call is the
 * same as the plain entry point of the same name.  dq_accum is [B,H,N,d]
 * fp32.  Other conventions as above.
 */
int attn_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse,
                 int B, int H, int Hkv, int N, int d, int causal, float scale, void* stream);
int attn_fwd_gqa_f16(const void* q, const void* k, const void* v, void* o, float* lse,
                     int B, int H, int Hkv, int N, int d, int causal, float scale, void* stream);
int attn_fwd_train_gqa(const void* q, const void* k, const void* v, void* o, float* o32,
                       float* lse, int B, int H, int Hkv, int N, int d, int causal, float scale,
                       void* stream);
int attn_fwd_train_gqa_f16(const void* q, const void* k, const void* v, void* o, float* o32,
                           float* lse, int B, int H, int Hkv, int N, int d, int causal,
                           float scale, void* stream);
int attn_bwd_preprocess_gqa(const void* q, const void* k, const void* v, const void* dO,
                            const float* lse, float* D, float* dq_accum, int B, int H, int Hkv,
                            int N, int d, int causal, float scale, void* stream);
int attn_bwd_preprocess_gqa_f16(const void* q, const void* k, const void* v, const void* dO,
                                const float* lse, float* D, float* dq_accum, int B, int H,
                                int Hkv, int N, int d, int causal, float scale, void* stream);
int attn_bwd_gqa(const void* q, const void* k, const void* v, const void* dO,
                 const float* lse, const float* D, float* dq_accum,
                 void* dq, void* dk, void* dv,
                 int B, int H, int Hkv, int N, int d, int causal, float scale, void* stream);
int attn_bwd_gqa_f16(const void* q, const void* k, const void* v, const void* dO,
                     const float* lse, const float* D, float* dq_accum,
                     void* dq, void* dk, void* dv,
                     int B, int H, int Hkv, int N, int d, int causal, float scale, void* stream);

/*
 * Grouped heads with the group split over CTAs.  attn_bwd_gqa runs one CTA
 * per (batch, K / V head, key block) that loops over all query heads of the
 * group, so with few K / V heads a few CTAs carry most of the work.  This
 * entry point gives each of `splits` CTAs per (batch, K / V head, key block)
 * H / Hkv / splits of the group's query heads; each writes its share of dK,
 * dV in fp32 to dkv_part, laid out [2][splits][B, Hkv, N, d] (dK shares,
 * then dV shares; caller-allocated, 16-byte aligned, 2 * splits * B * Hkv *
 * N * d floats), and a final pass sums the shares in split order and rounds
 * them to dk, dv (deterministic).  splits must divide H / Hkv; splits = 1 is
 * attn_bwd_gqa.  Dense layout; other arguments as for attn_bwd_gqa.
 * attn_gqa_split_hint returns the smallest split count whose heaviest CTA
 * does no more query-block iterations than the average SM (at most H / Hkv),
 * for the current device.
 */
int attn_bwd_gqa_split(const void* q, const void* k, const void* v, const void* dO,
                       const float* lse, const float* D, float* dq_accum, void* dq, void* dk,
                       void* dv, float* dkv_part, int splits, int B, int H, int Hkv, int N,
                       int d, int causal, float scale, void* stream);
int attn_bwd_gqa_split_f16(const void* q, const void* k, const void* v, const void* dO,
                           const float* lse, const float* D, float* dq_accum, void* dq, void* dk,
                           void* dv, float* dkv_part, int splits, int B, int H, int Hkv, int N,
                           int d, int causal, float scale, void* stream);
int attn_gqa_split_hint(int B, int H, int Hkv, int N, int causal);

/*
 * Packed variable-length batches, following the sj-techlog page ("2. module
 * 경계는 ..."): only the valid tokens are passed, concatenated, with
 * cu_seqlens (the cumulative token offset of each sequence) and the maximum
 * length, and softmax_lse is {batch, heads, seq_len}.
 *  - q, o, dO, dq: [total, H, d]; k, v, dk, dv: [total, Hkv, d] (16-bit,
 *    heads interleaved per token); o32, dq_accum: [total, H, d] fp32.
 *  - cu_seqlens: device int32 [B + 1], cu_seqlens[0] = 0, non-decreasing,
 *    cu_seqlens[B] = total; sequence b is tokens [cu_seqlens[b],
 *    cu_seqlens[b+1]).  Empty sequences are allowed.  Each sequence attends
 *    only to itself; the causal mask is per sequence (key j of a sequence is
 *    visible to its query i iff j <= i).  Grouped K / V heads as above.
 *  - lse: [B, H, max_seqlen] fp32, entries past a sequence's length are not
 *    written.  D: [total, H] fp32 (one value per packed row).
 *  - max_seqlen must be >= every length (the kernels clamp offsets to
 *    [0, total] and lengths to max_seqlen, so a bad cu_seqlens gives wrong
 *    results but no access outside the arrays); total = 0 enqueues nothing.
 *  - The training path is attn_fwd_train_varlen, then
 *    attn_bwd_preprocess_o32_varlen (D from the fp32 O), then attn_bwd_varlen.
 * Argument errors (null pointers, B < 1, total < 0, max_seqlen outside
 * 1..2^24, H not a multiple of Hkv, cu_seqlens not 4-byte aligned) return
 * ATTN_ERR_INVALID_ARG with nothing enqueued.  Other conventions as above.
 */
int attn_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                    const int* cu_seqlens, int B, int total, int max_seqlen, int H, int Hkv,
                    int d, int causal, float scale, void* stream);
int attn_fwd_varlen_f16(const void* q, const void* k, const void* v, void* o, float* lse,
                        const int* cu_seqlens, int B, int total, int max_seqlen, int H, int Hkv,
                        int d, int causal, float scale, void* stream);
int attn_fwd_train_varlen(const void* q, const void* k, const void* v, void* o, float* o32,
                          float* lse, const int* cu_seqlens, int B, int total, int max_seqlen,
                          int H, int Hkv, int d, int causal, float scale, void* stream);
int attn_fwd_train_varlen_f16(const void* q, const void* k, const void* v, void* o, float* o32,
                              float* lse, const int* cu_seqlens, int B, int total, int max_seqlen,
                              int H, int Hkv, int d, int causal, float scale, void* stream);
int attn_bwd_preprocess_o32_varlen(const float* o32, const void* dO, float* D, float* dq_accum,
                                   int total, int H, int d, void* stream);
int attn_bwd_preprocess_o32_varlen_f16(const float* o32, const void* dO, float* D,
                                       float* dq_accum, int total, int H, int d, void* stream);
int attn_bwd_varlen(const void* q, const void* k, const void* v, const void* dO,
                    const float* lse, const float* D, float* dq_accum,
                    void* dq, void* dk, void* dv, const int* cu_seqlens,
                    int B, int total, int max_seqlen, int H, int Hkv, int d, int causal,
                    float scale, void* stream);
int attn_bwd_varlen_f16(const void* q, const void* k, const void* v, const void* dO,
                        const float* lse, const float* D, float* dq_accum,
                        void* dq, void* dk, void* dv, const int* cu_seqlens,
                        int B, int total, int max_seqlen, int H, int Hkv, int d, int causal,
                        float scale, void* stream);

/*
 * Packed batches whose keys have lengths of their own (Lk != Lq per
 * sequence: a query chunk that attends to a longer key prefix, or queries
 * against a shorter set of keys).  The sj-techlog page's packed interface
 * (section "2. module 경계는 ...") passes one cu_seqlens and one max_s for q,
 * k and v together; the paldyn.com survey's version table ("v1에서 v3까지")
 * lists variable-length inputs among FlashAttention-2's additions.  Reading
 * taken here: queries and keys each get their own offsets and maximum.
 *  - q, o, dO, dq, o32, dq_accum: [total_q, H, d]; k, v, dk, dv:
 *    [total_k, Hkv, d].  Sequence b's queries are rows [cu_seqlens_q[b],
 *    cu_seqlens_q[b+1]) and its keys rows [cu_seqlens_k[b],
 *    cu_seqlens_k[b+1]) (both device int32 [B + 1], as cu_seqlens above).
 *  - Causal mask aligned bottom-right: with Lq queries and Lk keys, key j is
 *    visible to query i iff j <= i + Lk - Lq, so the last query sees every
 *    key.  With Lq = Lk this is the top-left mask of the other entry points.
 *    A query that sees no key (i < Lq - Lk) gets O = 0, lse = -inf and
 *    dQ = 0; keys of a sequence without queries get dK = dV = 0.
 *  - lse: [B, H, max_seqlen_q]; D: [total_q, H] (attn_bwd_preprocess_o32_varlen
 *    with total = total_q serves both paths).
 *  - max_seqlen_q / max_seqlen_k must be >= every query / key length.
 * Argument errors as for attn_fwd_varlen, plus a NULL or misaligned
 * cu_seqlens_k, total_k < 0 or max_seqlen_k outside 1..2^24.
 */
int attn_fwd_varlen_qk(const void* q, const void* k, const void* v, void* o, float* lse,
                       const int* cu_seqlens_q, const int* cu_seqlens_k, int B, int total_q,
                       int total_k, int max_seqlen_q, int max_seqlen_k, int H, int Hkv, int d,
                       int causal, float scale, void* stream);
int attn_fwd_varlen_qk_f16(const void* q, const void* k, const void* v, void* o, float* lse,
                           const int* cu_seqlens_q, const int* cu_seqlens_k, int B, int total_q,
                           int total_k, int max_seqlen_q, int max_seqlen_k, int H, int Hkv, int d,
                           int causal, float scale, void* stream);
int attn_fwd_train_varlen_qk(const void* q, const void* k, const void* v, void* o, float* o32,
                             float* lse, const int* cu_seqlens_q, const int* cu_seqlens_k, int B,
                             int total_q, int total_k, int max_seqlen_q, int max_seqlen_k, int H,
                             int Hkv, int d, int causal, float scale, void* stream);
int attn_fwd_train_varlen_qk_f16(const void* q, const void* k, const void* v, void* o, float* o32,
                                 float* lse, const int* cu_seqlens_q, const int* cu_seqlens_k,
                                 int B, int total_q, int total_k, int max_seqlen_q,
                                 int max_seqlen_k, int H, int Hkv, int d, int causal, float scale,
                                 void* stream);
int attn_bwd_varlen_qk(const void* q, const void* k, const void* v, const void* dO,
                       const float* lse, const float* D, float* dq_accum, void* dq, void* dk,
                       void* dv, const int* cu_seqlens_q, const int* cu_seqlens_k, int B,
                       int total_q, int total_k, int max_seqlen_q, int max_seqlen_k, int H,
                       int Hkv, int d, int causal, float scale, void* stream);
int attn_bwd_varlen_qk_f16(const void* q, const void* k, const void* v, const void* dO,
                           const float* lse, const float* D, float* dq_accum, void* dq, void* dk,
                           void* dv, const int* cu_seqlens_q, const int* cu_seqlens_k, int B,
                           int total_q, int total_k, int max_seqlen_q, int max_seqlen_k, int H,
                           int Hkv, int d, int causal, float scale, void* stream);

/*
 * Block-sparse layouts.  The sj-techlog page (section "대안, 비교와 선택
 * 기준") describes block-sparse FlashAttention: a block mask fixed in advance,
 * whose zero blocks are skipped.  Here the block is one 128 x 128 tile:
 *  - block_mask: device bytes, one per (query block r, key block c) with
 *    Nb = ceil(N / 128) blocks per side, row-major [Nb, Nb]; nonzero keeps the
 *    tile, zero drops it (its scores leave the softmax, as if -inf).  Head
 *    (b, h) reads the mask at block_mask + (b * H + h) * mask_head_stride;
 *    mask_head_stride = 0 shares one mask between all heads, otherwise it
 *    must be >= Nb * Nb.  The causal mask, if requested, applies on top.
 *  - A query row whose kept tiles hold no visible key has an empty softmax:
 *    its O row is 0, its lse -inf, and it contributes no gradient.  A key
 *    block that no query block keeps gets dK = dV = 0.
 *  - Dense [B,H,N,d] layout with one K / V head per query head (no grouped
 *    heads, no packed batches); N <= 49,152 (384 blocks).  Other arguments
 *    and errors as for attn_fwd / attn_fwd_train / attn_bwd; a bad mask
 *    argument returns ATTN_ERR_INVALID_ARG with nothing enqueued.
 *  - The training path is attn_fwd_train_bsparse, attn_bwd_preprocess_o32
 *    (D = rowsum(dO o O) from the fp32 O already holds only the kept tiles),
 *    then attn_bwd_bsparse with the same mask.  attn_bwd_preprocess (D from
 *    recomputed dense tiles) does not apply to a sparse layout.
 *  - Work and memory traffic scale with the number of kept tiles: a CTA
 *    lists its kept tiles in shared memory at start and visits only those
 *    (the forward's two query tiles per CTA visit the union of their kept
 *    key blocks; a tile that drops a listed block gives it P = 0).
 */
int attn_fwd_bsparse(const void* q, const void* k, const void* v, void* o, float* lse,
                     const void* block_mask, long long mask_head_stride, int B, int H, int N,
                     int d, int causal, float scale, void* stream);
int attn_fwd_bsparse_f16(const void* q, const void* k, const void* v, void* o, float* lse,
                         const void* block_mask, long long mask_head_stride, int B, int H, int N,
                         int d, int causal, float scale, void* stream);
int attn_fwd_train_bsparse(const void* q, const void* k, const void* v, void* o, float* o32,
                           float* lse, const void* block_mask, long long mask_head_stride, int B,
                           int H, int N, int d, int causal, float scale, void* stream);
int attn_fwd_train_bsparse_f16(const void* q, const void* k, const void* v, void* o, float* o32,
                               float* lse, const void* block_mask, long long mask_head_stride,
                               int B, int H, int N, int d, int causal, float scale, void* stream);
int attn_bwd_bsparse(const void* q, const void* k, const void* v, const void* dO,
                     const float* lse, const float* D, float* dq_accum, void* dq, void* dk,
                     void* dv, const void* block_mask, long long mask_head_stride, int B, int H,
                     int N, int d, int causal, float scale, void* stream);
int attn_bwd_bsparse_f16(const void* q, const void* k, const void* v, const void* dO,
                         const float* lse, const float* D, float* dq_accum, void* dq, void* dk,
                         void* dv, const void* block_mask, long long mask_head_stride, int B,
                         int H, int N, int d, int causal, float scale, void* stream);

/*
 * Combining partial results: the building blocks of attention over a
 * sequence whose keys and values are split into chunks (ring attention: the
 * paldyn.com survey "어텐션 비용 줄이기", section "다중 GPU 확장", has each
 * device keep its share of Q and pass K / V blocks around a ring, running the
 * single-device kernel on each pair).
 *
 * attn_merge merges a partial forward result into a running one, row by row,
 * in place: o_acc, o_part are [rows, d] fp32 outputs each normalised over its
 * own keys (the o32 of attn_fwd_train), lse_acc, lse_part [rows] their
 * natural-log logsumexps.  The merge is exact (sj-techlog "FlashAttention 원
 * 논문 해부", section "두 tile을 한 row로 합치는 식", written with normalised
 * outputs):
 *   L = log(exp(L_acc) + exp(L_part)),
 *   O = exp(L_acc - L) O_acc + exp(L_part - L) O_part,
 * with the larger statistic subtracted first; a side with L = -inf has
 * weight 0 and two of them give O = 0, L = -inf.  If o_out is not NULL the
 * merged O is also written there rounded to 16 bits ([rows, d]; bfloat16, or
 * IEEE half for the _f16 twin).  d is 64 or 128; o_acc, o_part, o_out
 * 16-byte aligned.  For [B,H,N,d] tensors rows = B*H*N.
 *
 * attn_convert writes y = scale * x rounded to 16 bits (the final cast of an
 * fp32 result such as a gradient summed over chunks).  elems must be a
 * multiple of 8; pointers 16-byte aligned.
 *
 * Both are element-wise passes over device memory; argument errors
 * return ATTN_ERR_INVALID_ARG (or _MISALIGNED / _UNSUPPORTED_HEAD_DIM) with
 * nothing enqueued, rows = 0 / elems = 0 enqueue nothing.
 */
int attn_merge(float* o_acc, float* lse_acc, const float* o_part, const float* lse_part,
               void* o_out, long long rows, int d, void* stream);
int attn_merge_f16(float* o_acc, float* lse_acc, const float* o_part, const float* lse_part,
                   void* o_out, long long rows, int d, void* stream);
int attn_convert(const float* x, void* y, long long elems, float scale, void* stream);
int attn_convert_f16(const float* x, void* y, long long elems, float scale, void* stream);

/*
 * Backward pass against one key / value chunk with fp32 dK, dV: as attn_bwd
 * (grouped heads allowed, Hkv as for attn_bwd_gqa), but instead of 16-bit dk,
 * dv it writes dk32, dv32 [B,Hkv,N,d] fp32, or adds to them when accumulate
 * is nonzero.  With lse and D of the whole rows (from the merged forward and
 * attn_bwd_preprocess_o32 of the merged fp32 O), the backward of a query
 * chunk against each key chunk yields that pair's share of the gradients
 * (the FlashAttention-2 review's "Backward Pass" with P = exp(S - lse)), so
 * the shares of dK, dV summed here over the query chunks, and of dQ summed in
 * dq_accum, are the gradients of the whole sequence, with no 16-bit rounding
 * of the partial sums.  dq is written from dq_accum after each call.
 * Dense layout only; dk32, dv32 16-byte aligned.
 */
int attn_bwd_acc(const void* q, const void* k, const void* v, const void* dO, const float* lse,
                 const float* D, float* dq_accum, void* dq, float* dk32, float* dv32,
                 int accumulate, int B, int H, int Hkv, int N, int d, int causal, float scale,
                 void* stream);
int attn_bwd_acc_f16(const void* q, const void* k, const void* v, const void* dO,
                     const float* lse, const float* D, float* dq_accum, void* dq, float* dk32,
                     float* dv32, int accumulate, int B, int H, int Hkv, int N, int d,
                     int causal, float scale, void* stream);

/*
 * Dropout on the attention probabilities, training path (sj-techlog page,
 * backward section: the forward keeps the pseudo-random generator's state,
 * and the backward regenerates the same dropout mask from it instead of
 * storing an N x N mask).  The generator is Philox4x32-10 (Salmon, Moraes,
 * Dror, Shaw, SC'11), written from its definition.
 *  - Mask: element (query i, key j) of (batch, head) index bh = b * H + h is
 *    kept iff byte j % 4 (bits 8 (j % 4) .. + 7) of output word i % 4 of
 *    Philox4x32-10 with counter (j / 4, i / 4, bh, offset) and key
 *    (seed mod 2^32, seed / 2^32) is below t = 256 (1 - p_drop) rounded half
 *    to even and clamped to [1, 256].  One generator call covers a 4 x 4
 *    patch.  t = 256 keeps everything (then identical to the plain entry
 *    points).  p_drop must be in [0, 1), else ATTN_ERR_INVALID_ARG.
 *  - Forward: O = (P o Z) V * 256 / t, with P the undropped softmax; lse is
 *    that of the undropped softmax; o32 as for attn_fwd_train (normalised by
 *    the sum of the rounded, undropped probabilities, then scaled).
 *  - Backward: D from attn_bwd_preprocess_o32 of that o32 (rowsum(dO o O));
 *    then with the same p_drop, seed and offset, dV = (P o Z)^T dO * 256 / t,
 *    dP = Z o (dO V^T) * 256 / t, dS = P o (dP - D), dQ = tau dS K,
 *    dK = tau dS^T Q.
 *  - Dense layout, one K / V head per query head.  Other conventions as for
 *    attn_fwd_train and attn_bwd.  Calls with another offset (or seed) draw
 *    an independent mask.
 */
int attn_fwd_train_dropout(const void* q, const void* k, const void* v, void* o, float* o32,
                           float* lse, float p_drop, unsigned long long seed, unsigned int offset,
                           int B, int H, int N, int d, int causal, float scale, void* stream);
int attn_fwd_train_dropout_f16(const void* q, const void* k, const void* v, void* o, float* o32,
                               float* lse, float p_drop, unsigned long long seed,
                               unsigned int offset, int B, int H, int N, int d, int causal,
                               float scale, void* stream);
int attn_bwd_dropout(const void* q, const void* k, const void* v, const void* dO,
                     const float* lse, const float* D, float* dq_accum, void* dq, void* dk,
                     void* dv, float p_drop, unsigned long long seed, unsigned int offset, int B,
                     int H, int N, int d, int causal, float scale, void* stream);
int attn_bwd_dropout_f16(const void* q, const void* k, const void* v, const void* dO,
                         const float* lse, const float* D, float* dq_accum, void* dq, void* dk,
                         void* dv, float p_drop, unsigned long long seed, unsigned int offset,
                         int B, int H, int N, int d, int causal, float scale, void* stream);

/* Static English description of a status code. */
const char* attn_status_string(int status);

/*
 * Synchronises `stream`, then reads and clears the device status word of the
 * current device.  Returns ATTN_OK, ATTN_ERR_TIMEOUT (a kernel gave up a
 * wait), or ATTN_ERR_DEVICE_FAULT (the synchronisation itself failed).
 */
int attn_get_device_status(void* stream);

/*
 * Self-test of the failure path: launches one tiny kernel that waits on a
 * barrier nothing ever completes, with a wait limit of about `timeout_us`
 * microseconds (1..1000000; the limit is a number of barrier polls, about
 * 2 us each).  The kernel records ATTN_ERR_TIMEOUT and returns; the GPU
 * context stays usable.  Returns ATTN_OK once enqueued.
 */
int attn_selftest_timeout(int timeout_us, void* stream);

/* Library version, for diagnostics. */
const char* attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* IO_AWARE_EXACT_GB300_ATTN_H */
