/*
 * fa.h -- C ABI of the GB300 (sm_103a) attention forward library
 *         (libfa_gb300.so, built from attention_forward_tma_gb300/csrc).
 *
 * The library computes, for every batch b, head h and query row i,
 *
 *     O_i   = sum_j softmax_j(scale * q_i . k_j) * v_j
 *     LSE_i = ln sum_j exp(scale * q_i . k_j)
 *
 * over the keys j the mask allows, streaming K/V blocks through shared memory
 * and keeping the score tile, the weight tile and the output accumulator in
 * tensor memory, so the score matrix never reaches global memory.
 *
 * Sources: "Flash Attention 4" (mlc.ai, Modern GPU Programming for MLSys),
 * sections "概览" (overview: O = softmax(QK^T/sqrt(d))V computed block by
 * block with per-row online-softmax state), "算法结构" (the update rule with
 * delayed rescaling at threshold 8), "重缩放与结果写回" (LSE = ln(row_sum) +
 * reference * scale, -inf for rows without a valid key) and "Causal Mask"
 * (bottom-right alignment). The explicit scale argument follows
 * "FlashAttention：一次前向计算" (qingsen), section "先看 attention 最后要得到什么",
 * which writes softmax(s * S) with s passed in rather than fixed.
 *
 * Conventions for every entry point below:
 *  - All tensor pointers are DEVICE pointers owned by the caller; the library
 *    never frees them and keeps no reference after the call returns.
 *  - bf16 / fp16 tensors are row-major with the head dimension d innermost and
 *    must be 16-byte aligned (TMA). d must be 64 or 128.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream). Work is
 *    enqueued asynchronously; argument errors are reported synchronously by the
 *    return value and enqueue nothing.
 *  - Nothing is printed and nothing is thrown across the ABI.
 *  - A device-side wait that exceeds its time limit makes the kernel give up
 *    cleanly (no trap, no hang) and records FA_ERR_TIMEOUT; read it with
 *    fa_last_device_status().
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, bad size, bad scale, bad cu_seqlens */
  FA_ERR_UNSUPPORTED = 2,  /* d not in {64,128}, device is not sm_103, kernel resources */
  FA_ERR_CUDA = 3,         /* a CUDA runtime/driver call failed (launch, tensor map, ...) */
  FA_ERR_TIMEOUT = 4,      /* a device-side wait gave up (reported by fa_last_device_status) */
  FA_ERR_NO_DEVICE = 5,    /* no CUDA device visible */
  FA_ERR_CAPACITY = 6      /* problem larger than the fixed scratch of fa_fwd_varlen_noalloc */
} fa_status;

/* Element type of q, k, v and o (all four share it). */
typedef enum { FA_DTYPE_BF16 = 0, FA_DTYPE_FP16 = 1 } fa_dtype;

/*
 * Fixed-length attention forward.
 *   q, k, v : bf16 [B, N, H, d]      (device, read only)
 *   o       : bf16 [B, N, H, d]      (device, written; rounded to nearest even)
 *   lse     : fp32 [B, H, N] or NULL (device, written: natural-log LSE of the
 *                                     scaled logits; -inf for a row with no key)
 *   B, H, N : >= 1;  d in {64, 128};  scale finite and > 0 (e.g. 1/sqrt(d))
 *   causal  : 0 = full attention; 1 = query i sees keys j <= i (bottom-right
 *             alignment, which is the usual lower-triangular mask since N_q = N_kv)
 * Returns FA_OK or an error code; the call is asynchronous on `stream`.
 */
int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
           int B, int H, int N, int d, float scale, int causal, void* stream);

/*
 * Grouped-query attention ("Flash Attention 4", section "GQA 支持"), and the
 * entry point for fp16 tensors.
 *   q, o    : [B, N, H, d]      k, v : [B, N, H_kv, d]    (dtype elements, device)
 *   lse     : fp32 [B, H, N] or NULL
 *   H_kv >= 1 must divide H (else FA_ERR_INVALID_ARG), and G = H / H_kv must
 *   divide 128, i.e. be a power of two up to 128 (else FA_ERR_UNSUPPORTED).
 *   Query head h attends with K/V head h / G; H_kv = H is multi-head attention.
 *   dtype   : FA_DTYPE_BF16 or FA_DTYPE_FP16; the weights P enter the second
 *             matrix product in that type, and o is written in it (round to
 *             nearest even).
 * Other arguments, errors and the mask as for fa_fwd;
 * fa_fwd(...) computes the same as fa_fwd_gqa(..., H_kv = H, ..., FA_DTYPE_BF16).
 * The kernel packs the G query heads of a group into the 128 rows of each Q
 * tile (128 / G positions x G heads), so every K/V block it loads serves the
 * whole group.
 */
int fa_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse,
               int B, int H, int H_kv, int N, int d, float scale, int causal, int dtype, void* stream);

/*
 * The general fixed-length entry point: N_q query rows and N_kv key rows per
 * sequence, grouped heads, bf16 / fp16, and an optional split of the keys.
 *   q, o : [B, N_q, H, d]      k, v : [B, N_kv, H_kv, d]     lse : fp32 [B, H, N_q] or NULL
 *   N_q, N_kv >= 1. causal = 1: query i sees keys j <= i + N_kv - N_q (bottom-right
 *   alignment, "Flash Attention 4", section "Causal Mask"); a row that sees no
 *   key (possible when N_q > N_kv) gets O = 0 and LSE = -inf.
 *   num_splits: the 128-key blocks of every sequence are cut into num_splits
 *   ranges (ceil(blocks / num_splits) blocks each) that run as separate tasks,
 *   each producing its normalised fp32 output and its LSE; a second kernel
 *   merges them: LSE = ln sum_s exp(LSE_s), O = sum_s exp(LSE_s - LSE) O_s
 *   ("FlashAttention：一次前向计算" (qingsen), the two-round example: partial
 *   results over key blocks merged through a common reference). This fills the
 *   GPU when B * H_kv * ceil(N_q * G / 256) is small and N_kv long (decoding).
 *   1 = no split; 0 = chosen by the library (split only when the unsplit tasks
 *   cannot fill the GPU); larger values are capped at the number of key blocks
 *   and at 128. With more than one range, partial results live in a temporary
 *   buffer of num_splits * B * N_q * H * (d + 1) * 4 bytes from the
 *   library's stream-ordered memory pool (cudaMallocFromPoolAsync / cudaFreeAsync on
 *   `stream`; the pool keeps its memory between calls).
 * Other arguments and errors as for fa_fwd_gqa.
 */
int fa_fwd_kv(const void* q, const void* k, const void* v, void* o, float* lse,
              int B, int H, int H_kv, int N_q, int N_kv, int d, float scale, int causal, int dtype,
              int num_splits, void* stream);

/*
 * One key shard of a longer sequence ("context" sharding of the keys, for example
 * over several GPUs): the attention of every query row over keys
 * [kv_offset, kv_offset + N_kv) of a sequence of N_kv_total keys, written as a
 * partial result for a later merge through the LSE (fa_lse_combine; the two-round
 * example of "FlashAttention：一次前向计算" merges the results of two key blocks
 * through a common reference, and "Flash Attention 4", section "重缩放与结果写回",
 * defines each part's LSE).
 *   q            : [B, N_q, H, d]        k, v : [B, N_kv, H_kv, d], the shard's keys
 *                  (dtype elements, device; H_kv, G and dtype as for fa_fwd_gqa)
 *   o_part       : fp32 [B, N_q, H, d] (device, written): the output normalised over
 *                  this shard's keys; 0 for a row that sees none of them
 *   lse_part     : fp32 [B, H, N_q] (device, written): natural-log LSE over this
 *                  shard's keys; -inf for a row that sees none of them
 *   N_kv_total   : keys of the whole sequence; kv_offset >= 0 and
 *                  kv_offset + N_kv <= N_kv_total (else FA_ERR_INVALID_ARG)
 *   causal       : 1 = the full sequence's bottom-right mask: query i sees global key
 *                  j <= i + N_kv_total - N_q, i.e. shard key jl <= i + N_kv_total - N_q
 *                  - kv_offset
 * Merging the shards of all ranges with fa_lse_combine (num_parts = number of
 * shards, parts stacked in the order of the o_parts / lse_parts layout) gives the
 * result of fa_fwd_kv over the whole sequence. No temporary memory; no key splits
 * inside the call. Other arguments and errors as for fa_fwd_kv.
 */
int fa_fwd_kv_partial(const void* q, const void* k, const void* v, float* o_part, float* lse_part,
                      int B, int H, int H_kv, int N_q, int N_kv, int N_kv_total, int kv_offset, int d,
                      float scale, int causal, int dtype, void* stream);

/*
 * Variable-length (packed) attention forward: sequence s owns the rows
 * [cu_seqlens[s], cu_seqlens[s+1]) of q, k, v and o; each sequence attends only
 * to itself (self-attention, causal mask aligned per sequence).
 *   q, k, v, o  : bf16 [total_tokens, H, d]  (device)
 *   lse         : fp32 [H, total_tokens] or NULL (device)
 *   cu_seqlens  : int32 [num_seqs + 1] (device), cu_seqlens[0] = 0,
 *                 non-decreasing, cu_seqlens[num_seqs] = total_tokens,
 *                 every length <= max_seqlen (zero-length sequences allowed)
 *   num_seqs >= 1, total_tokens >= 1, max_seqlen >= 1
 * Work tiles are ordered longest-first by a small schedule kernel launched on
 * the same stream ("FlashAttention-4（下）" (argus lesson 7), section "6. LPT 调度":
 * a pre-kernel sorts work tiles by their cost). Its tile list lives in a
 * temporary device buffer taken from the library's stream-ordered memory pool
 * (cudaMallocFromPoolAsync / cudaFreeAsync on `stream`; the pool keeps its memory
 * between calls).
 * The schedule kernel checks cu_seqlens on the device before it lists any tile
 * (cu_seqlens[0] = 0, non-decreasing, cu_seqlens[num_seqs] = total_tokens, every
 * length <= max_seqlen). If a rule is broken it lists no tile, so nothing is
 * written to o or lse, and fa_last_device_status returns FA_ERR_INVALID_ARG
 * (detail: 7 << 8 | the first offending sequence << 32). The general entry point
 * fa_fwd_varlen_kv checks cu_seqlens_kv the same way against total_kv (its key
 * lengths are not bounded by max_seqlen_kv, which only guides num_splits = 0).
 */
int fa_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                  const int* cu_seqlens, int num_seqs, int total_tokens, int max_seqlen,
                  int H, int d, float scale, int causal, void* stream);

/*
 * Variable-length grouped-query attention, bf16 or fp16:
 *   q, o : [total_tokens, H, d]      k, v : [total_tokens, H_kv, d]
 *   lse  : fp32 [H, total_tokens] or NULL
 * H_kv, G and dtype as for fa_fwd_gqa; everything else as for fa_fwd_varlen
 * (its temporary tile list holds H_kv * (ceil(total_tokens * G / 256) + num_seqs)
 * entries of 16 bytes). fa_fwd_varlen(...) computes the same as
 * fa_fwd_varlen_gqa(..., H_kv = H, ..., FA_DTYPE_BF16).
 */
int fa_fwd_varlen_gqa(const void* q, const void* k, const void* v, void* o, float* lse,
                      const int* cu_seqlens, int num_seqs, int total_tokens, int max_seqlen,
                      int H, int H_kv, int d, float scale, int causal, int dtype, void* stream);

/*
 * The general variable-length entry point: sequence s owns query rows
 * [cu_seqlens_q[s], cu_seqlens_q[s+1]) of q and o and key rows
 * [cu_seqlens_kv[s], cu_seqlens_kv[s+1]) of k and v (the two may be the same
 * array); its causal mask is bottom-right aligned on its own lengths, and a
 * sequence without keys gives O = 0, LSE = -inf for its rows.
 *   q, o : [total_q, H, d]     k, v : [total_kv, H_kv, d]     lse : fp32 [H, total_q] or NULL
 *   total_q, total_kv, max_seqlen_q >= 1; max_seqlen_kv >= 0 (only used to
 *   choose num_splits = 0); num_splits as for fa_fwd_kv (per sequence: its own
 *   key blocks are cut into num_splits ranges).
 * The temporary buffer holds the tile list (H_kv * (ceil(total_q * G / 256) +
 * num_seqs) * num_splits entries of 16 bytes) and, with more than one range,
 * the partial results (num_splits * total_q * H * (d + 1) * 4 bytes).
 */
int fa_fwd_varlen_kv(const void* q, const void* k, const void* v, void* o, float* lse,
                     const int* cu_seqlens_q, const int* cu_seqlens_kv, int num_seqs, int total_q,
                     int total_kv, int max_seqlen_q, int max_seqlen_kv, int H, int H_kv, int d, float scale,
                     int causal, int dtype, int num_splits, void* stream);

/*
 * The number of key ranges fa_fwd_kv / fa_fwd_varlen_kv would use for these
 * sizes (and, fixed length, this head dimension and mask: causal 0 or 1) on the
 * current device, given the same num_splits argument (0 = the library's choice:
 * for fixed length the count whose longest-first schedule of the tasks' key ranges
 * on the SMs, plus the merge of the partial results, is estimated shortest). With
 * *splits > 1 a call launches the merge kernel too.
 */
int fa_fwd_kv_splits(int B, int H, int H_kv, int N_q, int N_kv, int d, int causal, int num_splits, int* splits);
int fa_fwd_varlen_kv_splits(int num_seqs, int total_q, int max_seqlen_kv, int H, int H_kv, int num_splits,
                            int* splits);

/*
 * Merge of attention results computed over disjoint key sets (for example the
 * key ranges of one sequence held by different GPUs), through their LSE:
 *   LSE = ln sum_p exp(LSE_p),   O = sum_p exp(LSE_p - LSE) * O_p
 *   o_parts   : fp32 [num_parts, B, N, H, d]  (device; each part's normalised output)
 *   lse_parts : fp32 [num_parts, B, H, N]     (device; natural-log LSE, -inf = the part
 *                                              saw no key for that row: its O is not read)
 *   o         : [B, N, H, d] of dtype (bf16 / fp16), written
 *   lse       : fp32 [B, H, N] or NULL
 * A row whose parts are all -inf gets O = 0, LSE = -inf. Packed varlen rows
 * use B = 1, N = total rows (LSE layout [H, total]). d in {64, 128}.
 */
int fa_lse_combine(const float* o_parts, const float* lse_parts, int num_parts, int B, int N, int H, int d,
                   void* o, float* lse, int dtype, void* stream);

/*
 * fa_fwd_varlen_noalloc: the same computation, arguments and results as
 * fa_fwd_varlen, for callers that cannot allocate device memory at call time:
 * for example a serving process that hands all of the GPU's memory to its own
 * pool at start-up (so a later cudaMalloc fails), or a latency-critical loop
 * that must not run allocator calls, which can block on other work of the
 * device. The paper has no counterpart; this entry point exists only for
 * such callers.
 *
 * It allocates nothing. Its work-tile list lives in a fixed array of this
 * library (2 MiB + 16 bytes of device memory, taken on every GPU that loads
 * the library and kept until the process exits), so:
 *  - the problem must satisfy H * (ceil(total_tokens / R) + num_seqs) <= 131072,
 *    R the query rows per work tile: 256, or 128 when the library runs one-tile
 *    tasks (FA_OPT_SOLO_TILES = 1 forces them; the automatic choice takes them only
 *    for problems of at most one tile per SM), else it returns FA_ERR_CAPACITY
 *    and enqueues nothing;
 *  - all calls on a device share that array: calls whose work overlaps on the
 *    GPU (for example on two streams at once) race and may return wrong
 *    results; order them on one stream or with events;
 *  - nothing in the array needs clearing between calls: each call's schedule
 *    kernel overwrites the tile count and every tile it reports;
 *  - the first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress) with that device current; make that first call
 *    before any stream capture.
 */
int fa_fwd_varlen_noalloc(const void* q, const void* k, const void* v, void* o, float* lse,
                          const int* cu_seqlens, int num_seqs, int total_tokens, int max_seqlen,
                          int H, int d, float scale, int causal, void* stream);

/*
 * Backward pass of fa_fwd_kv without key splits: gradients of
 * O = softmax(scale * Q K^T) V for an upstream gradient dO ("FlashAttention-4（下）"
 * (argus lesson 7), section 1: S and P are recomputed from Q, K and the forward's
 * LSE; dV = P^T dO, dP = dO V^T, dS = P * (dP - rowsum(dO * O)), dQ = scale * dS K,
 * dK = scale * dS^T Q; with grouped heads dK and dV of a K/V head sum over its G
 * query heads).
 *   q, o, dout, dq : [B, N_q, H, d]      k, v, dk, dv : [B, N_kv, H_kv, d]
 *                    (dtype elements, device; dq, dk, dv written)
 *   lse            : fp32 [B, H, N_q], the LSE that fa_fwd* wrote for these q, k, v
 *   other arguments as for fa_fwd_kv (bottom-right causal mask).
 * dQ is accumulated over key blocks in fp32 by reduce-adds in arrival order, so
 * its last bits may differ from run to run unless FA_OPT_BWD_DETERMINISTIC is set;
 * dK and dV are always deterministic. A temporary buffer of B*N_q*H*d*4 +
 * 2*B*H_kv*ceil(N_q*G/128)*128*4 + 256 bytes (+ 4 bytes per 128-row Q tile in the
 * deterministic mode) comes from the library's stream-ordered memory pool
 * (cudaMallocFromPoolAsync / cudaFreeAsync on `stream`; memory kept between calls). One CTA per SM walks the tasks (key block of a
 * (batch, K/V head) pair) in order, claiming the next from a counter in that buffer.
 */
int fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
           void* dq, void* dk, void* dv, int B, int H, int H_kv, int N_q, int N_kv, int d, float scale,
           int causal, int dtype, void* stream);

/*
 * Backward pass of fa_fwd_varlen_kv without key splits (same gradients as fa_bwd,
 * per sequence): sequence s has query rows [cu_seqlens_q[s], cu_seqlens_q[s+1]) and
 * key rows [cu_seqlens_kv[s], cu_seqlens_kv[s+1]), with its own bottom-right causal
 * diagonal; rows of one sequence never see another's keys.
 *   q, o, dout, dq : [total_q, H, d]     k, v, dk, dv : [total_kv, H_kv, d]
 *                    (dtype elements, device; dq, dk, dv written)
 *   lse            : fp32 [H, total_q], the LSE that fa_fwd_varlen* wrote
 *   cu_seqlens_q, cu_seqlens_kv : device int32 [num_seqs + 1], non-decreasing, starting
 *                    at 0 and ending at total_q / total_kv, every length at most
 *                    max_seqlen_q / max_seqlen_kv; empty sequences are allowed (a query
 *                    row without keys gets dQ = 0, a key without queries dK = dV = 0).
 *                    A one-block kernel checks the arrays on the device before any other
 *                    work: if they break a rule, the call writes nothing to dq, dk, dv and
 *                    fa_last_device_status returns FA_ERR_INVALID_ARG (detail: 7 << 8 |
 *                    the first offending sequence << 32)
 *   max_seqlen_q, max_seqlen_kv : the longest sequence's lengths (upper bounds suffice;
 *                    they size the grid and the packed-row buffers)
 *   other arguments as for fa_bwd. Errors: as fa_bwd, plus FA_ERR_INVALID_ARG for null
 *   or misaligned cu_seqlens, num_seqs, totals or maxima <= 0. The temporary buffer is
 *   total_q*H*d*4 + 2*num_seqs*H_kv*ceil(max_seqlen_q*G/128)*128*4 bytes (+ the
 *   deterministic mode's counters), from the library's stream-ordered memory pool.
 */
int fa_bwd_varlen(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                  void* dq, void* dk, void* dv, const int* cu_seqlens_q, const int* cu_seqlens_kv, int num_seqs,
                  int total_q, int total_kv, int max_seqlen_q, int max_seqlen_kv, int H, int H_kv, int d,
                  float scale, int causal, int dtype, void* stream);

/* Text for a status code (static storage; never NULL). */
const char* fa_error_string(int status);

/*
 * Synchronizes `stream`, then returns and clears the device-side status word of
 * the current device: FA_OK; FA_ERR_TIMEOUT if a kernel of this library gave up
 * on a wait since the last call; FA_ERR_INVALID_ARG if a varlen call's device-side
 * check rejected its cu_seqlens (FA_ERR_CUDA if the synchronization failed).
 * If `detail` is not NULL it receives the raw word: code | role << 8 | barrier << 16
 * | block << 32 (role 7 = the cu_seqlens check, its "block" the first offending
 * sequence).
 */
int fa_last_device_status(void* stream, unsigned long long* detail);

/*
 * Process-wide tuning knobs (not thread-safe; meant for tests and benchmarks).
 *   FA_OPT_TAU             : rescale threshold tau in base-2 exponent units (default 8);
 *                            fp16 calls use min(tau, 15) so the weights P <= 2^tau
 *                            stay finite in fp16
 *   FA_OPT_WAIT_TIMEOUT_NS : device wait limit in nanoseconds (default 2e9)
 *   FA_OPT_PERSISTENT      : task scheduling. 2 = one CTA per task in launch order, and
 *                            each running CTA takes over the tasks of CTAs not yet
 *                            launched (cluster launch control; the default);
 *                            1 = one CTA per SM with a static task stride;
 *                            0 = one CTA per task, no take-over; -1 = restore the default.
 *                            fa_bwd / fa_bwd_varlen: 0 = one CTA per task; any other
 *                            value = one CTA per SM claiming tasks in order (default)
 *   FA_OPT_EXP2_EMULATION  : number of 16-element groups per 128-wide row (0..8)
 *                            whose exp2 is evaluated with the FMA polynomial instead
 *                            of the hardware ex2 unit (default 0)
 *   FA_OPT_BWD_DETERMINISTIC : 1 = fa_bwd adds the dQ contributions of the key blocks
 *                            of every Q tile in one fixed order (key block 0 first),
 *                            so dQ is bitwise reproducible ("FlashAttention-4（下）"
 *                            section 5, deterministic mode: a semaphore per tile
 *                            serialises the global accumulation); key blocks wait for
 *                            their predecessors, which costs speed. 0 = arrival order
 *                            (default).
 *   FA_OPT_SOFTMAX_STAGGER : 1 = the two softmax warpgroups of the forward take turns at
 *                            their exponential phases, so they never compete for the
 *                            exp2 unit at once ("Flash Attention 4", section on the
 *                            differences between the paper and the TIRx kernel: the
 *                            paper's ordering of the two softmax warpgroups).
 *                            0 = no ordering (default).
 *   FA_OPT_STATS_TMEM      : 1 = the forward's per-block rescale factor acc_scale goes
 *                            from the softmax warpgroup to the correction warpgroup
 *                            through tensor memory (a free column of the score tile)
 *                            instead of a shared-memory mailbox (same section: the
 *                            paper passes the statistics through spare TMEM);
 *                            default 1. 0 = shared memory.
 *   FA_OPT_BWD_SECTION     : (sequence, K/V head) pairs per L2 section of the backward's
 *                            grid order (whole number; 0 = the library's choice, about
 *                            512 CTAs per section)
 *   FA_OPT_SOLO_TILES      : fixed-length forward tasks of one 128-row Q tile whose score
 *                            tile alternates between the two S buffers of tensor memory,
 *                            so a block's QK^T overlaps the previous block's softmax
 *                            (instead of two Q tiles sharing each K/V block). -1 = the
 *                            library's choice (default: when the 256-row tasks leave SMs
 *                            idle and the 128-row ones fit in one wave, e.g. decoding and
 *                            small batches; for varlen calls the rule takes an upper bound
 *                            of the work tiles), 0 = never, 1 = always.
 * The forward variants compute the same result as the default path.
 * Returns FA_OK or FA_ERR_INVALID_ARG.
 */
enum { FA_OPT_TAU = 1, FA_OPT_WAIT_TIMEOUT_NS = 2, FA_OPT_PERSISTENT = 3, FA_OPT_EXP2_EMULATION = 4,
       FA_OPT_BWD_DETERMINISTIC = 5, FA_OPT_SOFTMAX_STAGGER = 6, FA_OPT_STATS_TMEM = 7,
       FA_OPT_BWD_SECTION = 8, FA_OPT_SOLO_TILES = 9 };
int fa_set_option(int option, double value);

/*
 * Hand the library's cached temporary memory back to the system. The split
 * partials, the varlen tile list and the backward's workspace come from a
 * stream-ordered pool that keeps its memory between calls (so that a caller
 * which synchronises every step does not map it again each time); after a very
 * large call that can be gigabytes (the backward's fp32 dQ accumulator is
 * 4 * B * N_q * H * d bytes). This releases, on every device the library has
 * used, the pool memory not backing an allocation still pending on a stream:
 * call it once the streams that ran the library's calls have been synchronised.
 * Returns FA_OK (also when no pool exists yet), or FA_ERR_CUDA.
 */
int fa_release_cached_memory(void);

/* Library version, as major*10000 + minor*100 + patch. */
int fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H */
