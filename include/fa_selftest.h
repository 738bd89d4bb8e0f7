/*
 * fa_selftest.h -- diagnostic entry points of libfa_gb300.so.
 *
 * These calls exercise single pieces of the attention kernel on the GPU so a
 * test can check each against a plain host computation: the tcgen05 MMA
 * plumbing on one tile, the exponential paths, the bounded waits, and the
 * varlen longest-first schedule. They are not needed to run attention.
 * Conventions as in fa.h: device pointers owned by the caller, `stream` is a
 * cudaStream_t, return value is an fa_status code.
 */
#ifndef FA_GB300_SELFTEST_H
#define FA_GB300_SELFTEST_H

#ifdef __cplusplus
extern "C" {
#endif

/*
 * One tile through the kernel's own TMA maps, shared-memory descriptors and
 * tcgen05 instructions:
 *   s_out = Q K^T          (fp32 [128, 128])    q, k : [128, d]
 *   o_out = P V            (fp32 [128, d])      p : [128, 128], v : [128, d]
 * q, k, v, p in the element type dtype (FA_DTYPE_BF16 or FA_DTYPE_FP16 of fa.h).
 * d in {64, 128}. Synchronizes the stream before returning.
 */
int fa_selftest_mma_tile(const void* q, const void* k, const void* v, const void* p,
                         float* s_out, float* o_out, int d, int dtype, void* stream);

/* y[i] = 2^x[i] with the hardware ex2 unit (use_poly = 0), with the FMA
 * polynomial used for part of the softmax exponentials (use_poly = 1), or with
 * the packed-pair (f32x2) form of that polynomial the softmax runs (use_poly = 2).
 * x, y: fp32 [n] device. Asynchronous. */
int fa_selftest_exp2(const float* x, float* y, int n, int use_poly, void* stream);

/* Launches a kernel whose only mbarrier wait can never complete, with the given
 * wait limit; the wait must give up without trapping or hanging. Synchronizes
 * the stream and returns the recorded status: FA_ERR_TIMEOUT is the expected
 * (correct) outcome, FA_OK would mean the wait did not time out. */
int fa_selftest_wait_timeout(unsigned long long timeout_ns, void* stream);

/* The varlen longest-first tile schedule that fa_fwd_varlen_kv computes,
 * written to caller buffers: tasks = int32 [capacity, 4] of {sequence, K/V
 * head | key range << 16, m_block, cost in K/V blocks}, sorted by
 * non-increasing cost; *count = number written. group = G, the query heads per
 * K/V head (1 for fa_fwd_varlen; a power of two up to 128): a sequence of L_q
 * query rows has L_q * G packed rows, cut into m_blocks of 256 rows, and row r
 * of an m_block is position r / G. splits = key ranges per tile (1..128).
 * cu_seqlens_q / cu_seqlens_kv: device int32 [num_seqs + 1]. Asynchronous. */
int fa_varlen_schedule(const int* cu_seqlens_q, const int* cu_seqlens_kv, int num_seqs, int H_kv, int group,
                       int causal, int splits, int capacity, void* tasks, int* count, void* stream);

/*
 * Pipeline tracing. Only the tracing build of the library (compiled with
 * -DFA_TRACE, libfa_gb300_trace.so) records; the normal build returns
 * FA_ERR_UNSUPPORTED from fa_trace_configure.
 * fa_trace_configure(buf, ctas): later fa_fwd / fa_fwd_varlen calls make one
 * leader thread per role of CTAs 0..ctas-1 stamp clock64 at each pipeline
 * hand-off into buf (device, uint64 [ctas][roles][slots]); ctas = 0 turns it
 * off. Per role, word 0 is the number of events, then each event is two
 * words: the SM clock and (event code << 32 | K/V block index). Roles:
 * 0 TMA producer, 1 MMA issuer, 2 softmax of Q tile 0, 3 softmax of Q tile 1,
 * 4 correction/epilogue. The forward also adds, over every CTA, the softmax rows'
 * updates from a later key block (word ctas * roles * slots) and those of them that
 * moved the row's reference and rescaled O (the word after it). The buffer must hold
 * ctas * roles * slots + 2 words, zeroed by the caller.
 * fa_trace_layout reports roles and slots per role (works in both builds).
 */
int fa_trace_configure(void* buf, int ctas);
int fa_trace_layout(int* roles, int* slots_per_role);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_SELFTEST_H */
