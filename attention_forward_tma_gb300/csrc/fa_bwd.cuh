// fa_bwd.cuh -- the attention backward pass for GB300 (sm_103a).
//
// Gradients of O = softmax(s * Q K^T) V for an upstream dO ("FlashAttention-4（下）"
// (argus lesson 7), section 1: recompute S and P, then the products for dV, dP,
// dK and dQ with the elementwise softmax gradient between them):
//
//   P  = exp2(S * s * log2 e - LSE * log2 e)    (S = Q K^T recomputed, LSE from the forward)
//   dV += P^T dO          dP = dO V^T          dS = s * P * (dP - D),  D = rowsum(dO * O)
//   dK += dS^T Q          dQ += dS K
//
// A task is one block of 128 keys of one (sequence, K/V head): it walks over the
// 128-row Q tiles that can see the block, accumulating dK and dV in tensor memory
// (section 2 of the same page: TMEM accumulators let several products be in
// flight). CTAs of 512 threads, one per SM, claim the tasks in order and run them
// back to back (see the kernel). S and P are computed transposed (S^T = K Q^T, keys on
// the TMEM lanes), so P^T is already the A operand of the dV product, as the page
// describes. dQ of each (Q tile, key block) pair is added to an fp32 buffer in
// global memory (section 4: the dQ sum over key blocks is a global atomic
// accumulation): staged in shared memory and sent as TMA reduce-adds, 16 KB per
// operation, in place of per-thread atomics. With grouped heads the Q tiles hold
// the packed (position, query head) rows of the forward, so every query head of the
// group contributes to the task's dK and dV without atomics.
//
// Roles: WG0 and WG1 (warps 0-7, one thread per key row) compute P and dS for
// query columns 0-63 and 64-127 of the tile (the LSE is known, so the halves need
// no exchange); WG2 (warps 8-11, one thread per Q-tile row) moves dQ from TMEM
// into shared memory and issues its reduce-adds, and at the end writes dV; warp 12
// issues the TMA loads (Q, dO and the tile's base-2 LSE and D), warp 13 the
// tcgen05 MMAs. WG0 and WG1 write the two halves of dK at the end.
//
// Tensor memory (512 columns): dV [0, d), dK [128, 128+d), S^T [256, 384) with P^T
// as 16-bit pairs over the upper 32 columns of each 64-column half, dP^T [384, 512)
// -- reused for dQ once dS is in shared memory. Shared memory (226 KB of the 227 KB a CTA may have):
// K, V, two stages of (Q, dO, LSE, D), and the dS tile (128 keys x 128 rows,
// 128-byte swizzle): the same bytes are the K-major A operand of dK (M = keys)
// and the MN-major A operand of dQ (M = rows). Once a step's products are done,
// its Q and dO buffers hold the staged fp32 dQ tile for the reduce-adds.
//
// Every wait is bounded as in the forward kernel.
#pragma once

#include <climits>
#include <cuda_fp16.h>

#include "fa_fwd.cuh"

namespace fa {

constexpr int kBwdThreads = 512;

struct BwdParams {
  CUtensorMap tm_q, tm_do;   // [tokens_q, H, d]: box 64 x G x 128/G (one packed 128-row tile)
  CUtensorMap tm_k, tm_v;    // [tokens_k, H_kv, d]: box 64 x 1 x 128
  CUtensorMap tm_dq;         // fp32 dq_acc [tokens_q, H, d]: box 32 x G x 128/G, reduce-adds
  const float* lse2;         // [B, H_kv, mpad], packed rows: forward LSE * log2(e)
  const float* dsum;         // [B, H_kv, mpad], packed rows: D = rowsum(dO * O)
  // variable length (both null for fixed length): B = number of sequences, sequence b
  // has query rows [cu_q[b], cu_q[b+1]) and key rows [cu_k[b], cu_k[b+1]); Nq, Nk,
  // mpad and nkb are then those of the longest sequence (grid and packed-row stride)
  const int* cu_q;
  const int* cu_k;
  float* dq_acc;             // fp32 [tokens_q, H, d]; zero on entry
  uint16_t* dk;              // [tokens_k, H_kv, d]
  uint16_t* dv;              // [tokens_k, H_kv, d]
  int B, H, Hkv, gshift, Nq, Nk;
  int nkb;                   // 128-key blocks per sequence
  int section;               // (sequence, K/V head) pairs per L2 section of the grid order
  int mpad;                  // packed rows per (b, K/V head), rounded up to 128
  int num_tasks;
  float scale, scale_log2;
  unsigned long long timeout_ns;
  unsigned long long* trace;     // tracing build only: clock stamps per CTA and role (else null)
  int trace_ctas;
  // deterministic dQ: per (b, kv head, Q tile) the number of key blocks that have
  // added their dQ so far (zero on entry); key block j adds only after blocks
  // 0 .. j-1 did, so every dQ element is summed in one fixed order. Null: no order.
  int* sem;
  int ntiles;
  int* task_counter;         // zero on entry: tasks claimed beyond the first gridDim.x
  const int* cu_ok;          // variable length: 1 if cu_q / cu_k passed fa_bwd_check_cu_kernel (else
                             // every kernel of the call returns at once); null for fixed length
};

template <int D>
struct BwdLayout {
  static_assert(D == 64 || D == 128, "head dim");
  static constexpr int kHalves = D / 64;
  static constexpr int kSlab = 128 * 128;            // 128 rows x 128 bytes
  static constexpr int kTile = kHalves * kSlab;       // 128 rows x D, 16-bit
  static constexpr int kK = 0, kV = kTile, kQ = 2 * kTile, kDO = 4 * kTile, kDS = 6 * kTile;
  static constexpr int kStats = kDS + 2 * kSlab;      // dS: 128 keys x 128 rows
  static constexpr int kStatsBytes = 1024;            // per stage: 128 base-2 LSE, then 128 D (fp32)
  static constexpr int kBar = kStats + 2 * kStatsBytes;
  enum : int {
    bKV = 0, bQFull = 1, bQEmpty = 3, bSFull = 5, bPReady = 6, bdPFull = 7, bdPEmpty = 8, bdSReady = 9,
    bdSEmpty = 10, bdQFull = 11, bFinal = 12, bDrain = 13, bdQStaged = 14, bAccFree = 15, bTaskFull = 16,
    bTaskEmpty = 18, kNumBars = 20
  };
  static constexpr int kTaskReaders = 13;              // warps that read a claimed task: MMA, WG0-2
  static constexpr int kMisc = kBar + 256;
  static constexpr int kBytes = kMisc + 64;
  static constexpr int kAlloc = kBytes;               // the dynamic shared memory is 1024-byte aligned
  static_assert(kNumBars * 8 <= 256, "barriers");
  static_assert(kAlloc <= 227 * 1024, "shared memory per CTA");
  static constexpr uint32_t cDV = 0, cDK = 128, cS = 256, cDP = 384;
};

// Byte offset of K step kk (16 elements) in a K-major, 128-byte-swizzled operand
// made of 64-element slabs of 128 rows.
template <int SLAB>
__device__ __forceinline__ uint32_t kmajor_step(int kk) {
  return (uint32_t)((kk / 4) * SLAB + (kk % 4) * 32);
}

__device__ __forceinline__ float half_bits_to_f32(uint16_t x, bool f16) {
  return f16 ? __half2float(__ushort_as_half(x)) : __uint_as_float((uint32_t)x << 16);
}

// ------------------------------------------------------------------ preprocessing
// D / 8 lanes per (query row, head) of the [tokens, H, d] tensors (16-byte loads):
// D = rowsum(dO * O) in fp32 and the forward's LSE in base 2, both written at the row's packed index
// (sequence, kv head, position * G + head % G); the row of the fp32 dQ accumulator is
// zeroed on the way. Fixed length: sequence b holds rows [b * Nq, (b + 1) * Nq) and the
// LSE is [B, H, Nq]; variable length (cu_q not null): the sequence of a row is found by
// bisection in cu_q[0 .. B] and the LSE is [H, tokens].
template <int D, bool F16>
__global__ void __launch_bounds__(256) fa_bwd_pre_kernel(const uint16_t* __restrict__ o,
                                                         const uint16_t* __restrict__ dout,
                                                         const float* __restrict__ lse, float* __restrict__ lse2,
                                                         float* __restrict__ dsum, float* __restrict__ dq_acc,
                                                         long long tokens, const int* __restrict__ cu_q, int B,
                                                         int H, int gshift, int Nq, int mpad,
                                                         const int* __restrict__ cu_ok) {
  if (cu_ok != nullptr && *cu_ok == 0) return;
  constexpr int kLanes = D / 8;                // lanes per row: 16-byte loads of 8 elements
  constexpr int kRowsPerWarp = 32 / kLanes;
  const int lane = threadIdx.x & 31;
  const long long w = ((long long)blockIdx.x * 8 + (threadIdx.x >> 5)) * kRowsPerWarp + lane / kLanes;
  const int part = lane % kLanes;
  const bool valid = w < tokens * H;
  float acc = 0.f;
  if (valid) {
    const uint4 ov = *reinterpret_cast<const uint4*>(o + w * D + part * 8);
    const uint4 gv = *reinterpret_cast<const uint4*>(dout + w * D + part * 8);
    float4* z = reinterpret_cast<float4*>(dq_acc + w * D + part * 8);
    z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
    z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
    const uint32_t ow[4] = {ov.x, ov.y, ov.z, ov.w}, gw[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      acc = fmaf(half_bits_to_f32((uint16_t)(ow[e] & 0xffffu), F16), half_bits_to_f32((uint16_t)(gw[e] & 0xffffu), F16),
                 acc);
      acc = fmaf(half_bits_to_f32((uint16_t)(ow[e] >> 16), F16), half_bits_to_f32((uint16_t)(gw[e] >> 16), F16), acc);
    }
  }
#pragma unroll
  for (int x = kLanes / 2; x > 0; x >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, x);
  if (valid && part == 0) {
    const int h = (int)(w % H);
    const long long bp = w / H;
    int b, pos;
    size_t li;
    if (cu_q == nullptr) {
      b = (int)(bp / Nq);
      pos = (int)(bp % Nq);
      li = ((size_t)b * H + h) * Nq + pos;
    } else {
      int lo = 0, hi = B;   // the last sequence starting at or before the row
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (cu_q[mid] <= bp) lo = mid; else hi = mid;
      }
      b = lo;
      pos = (int)(bp - cu_q[lo]);
      li = (size_t)h * tokens + bp;
    }
    const int Hkv = H >> gshift;
    const size_t idx = ((size_t)b * Hkv + (h >> gshift)) * mpad + ((size_t)pos << gshift) + (h & ((1 << gshift) - 1));
    dsum[idx] = acc;
    lse2[idx] = lse[li] * 1.4426950408889634f;
  }
}

// dQ (16-bit) from the fp32 accumulator, 4 elements per thread.
template <bool F16>
__global__ void __launch_bounds__(256) fa_bwd_post_kernel(const float4* __restrict__ acc, uint2* __restrict__ dq,
                                                          long long n4, const int* __restrict__ cu_ok) {
  if (cu_ok != nullptr && *cu_ok == 0) return;
  const long long i = (long long)blockIdx.x * 256 + threadIdx.x;
  if (i >= n4) return;
  const float4 x = acc[i];
  dq[i] = make_uint2(pack_16x2<F16>(x.x, x.y), pack_16x2<F16>(x.z, x.w));
}

// Check of the sequence offsets of a variable-length backward call, one CTA:
// cu_q[0] = cu_k[0] = 0, both non-decreasing, cu_q[B] = total_q, cu_k[B] = total_k,
// every query length <= max_q and every key length <= max_k (the grid and the packed
// LSE / D rows are sized by the longest sequences). *ok = 1 if all hold; else *ok
// stays 0 and FA_ERR_INVALID_ARG | 7 << 8 | (first offending sequence) << 32 is
// recorded in the device status word.
__global__ void __launch_bounds__(1024) fa_bwd_check_cu_kernel(const int* __restrict__ cu_q,
                                                               const int* __restrict__ cu_k, int B, int total_q,
                                                               int total_k, int max_q, int max_k, int* ok) {
  __shared__ int first_bad;
  if (threadIdx.x == 0) first_bad = INT_MAX;
  __syncthreads();
  auto entry_ok = [&](const int* cu, int s, int total, int max_len) {
    const int a = cu[s], b = cu[s + 1];
    return b >= a && (s != 0 || a == 0) && (s != B - 1 || b == total) && b - a <= max_len;
  };
  for (int s = threadIdx.x; s < B; s += blockDim.x)
    if (!entry_ok(cu_q, s, total_q, max_q) || !entry_ok(cu_k, s, total_k, max_k)) atomicMin(&first_bad, s);
  __syncthreads();
  if (threadIdx.x == 0) {
    if (first_bad == INT_MAX) {
      *ok = 1;
    } else {
      *ok = 0;
      atomicCAS(&g_fa_status, 0ull, 1ull | (7ull << 8) | ((unsigned long long)(uint32_t)first_bad << 32));
    }
  }
}

// ------------------------------------------------------------------ tasks
// A task is key block j of one (sequence, kv head) pair. Task indices run in sections
// of p.section pairs, so that the CTAs in flight share Q, dO and the fp32 dQ
// accumulator rows in L2; inside a section key block j of every pair comes before
// block j+1 (heavy blocks, small j under the causal mask, first; and block j of a pair
// always after block j-1, which the deterministic mode's ordered dQ additions rely on).
struct BwdTask {
  int b, kvh, j;
  int Nq, Nk, tok_q, tok_k;   // the sequence's lengths and first rows
  int off;                    // bottom-right causal offset Nk - Nq
  int i0, n;                  // its Q tiles: i0 .. i0 + n - 1
  bool skip;                  // a shorter sequence of a varlen batch: no such key block
};

template <bool CAUSAL>
__device__ __forceinline__ BwdTask bwd_task(const BwdParams& p, int idx) {
  BwdTask t;
  const int pairs = p.B * p.Hkv;
  const int per_sec = p.section * p.nkb;
  const int sec = idx / per_sec, rem = idx - sec * per_sec;
  const int in_sec = min(p.section, pairs - sec * p.section);   // the last section may be smaller
  t.j = rem / in_sec;
  const int bh = sec * p.section + (rem - t.j * in_sec);
  t.b = bh / p.Hkv;
  t.kvh = bh - t.b * p.Hkv;
  t.Nq = p.Nq;
  t.Nk = p.Nk;
  t.tok_q = t.b * p.Nq;
  t.tok_k = t.b * p.Nk;
  if (p.cu_q != nullptr) {
    t.tok_q = p.cu_q[t.b];
    t.Nq = p.cu_q[t.b + 1] - t.tok_q;
    t.tok_k = p.cu_k[t.b];
    t.Nk = p.cu_k[t.b + 1] - t.tok_k;
  }
  t.skip = t.j * 128 >= t.Nk;
  t.off = t.Nk - t.Nq;
  const int ntiles = ((t.Nq << p.gshift) + 127) / 128;
  t.i0 = 0;
  if (CAUSAL) {
    const long long pmin = (long long)t.j * 128 - t.off;   // the first position that sees key j*128
    if (pmin > 0) t.i0 = (int)min((long long)ntiles, (pmin << p.gshift) / 128);
  }
  t.n = t.skip ? 0 : ntiles - t.i0;
  return t;
}

// ------------------------------------------------------------------ the main kernel
// Persistent: CTA c starts with task c; when its producer warp has issued the loads of
// a task it claims the next one from a global counter (tasks gridDim.x, gridDim.x + 1,
// ... in task order: a CTA that is free first takes the next heaviest task) and hands
// it to the other warps through a two-slot ring (b_task_full / b_task_empty). Claims
// only grow, so a task waits only on tasks claimed before it (the deterministic mode's
// ordered dQ additions cannot deadlock). Every per-step barrier phase follows a step
// counter g that runs on across the CTA's tasks, so the next task's first loads and
// products overlap the previous task's last dQ additions and its dK / dV write-out:
// the next K, V wait only for the previous task's last products (b_final), the next
// dV / dK only for the write-out's reads of their tensor-memory columns (b_acc_free).
template <int D, bool CAUSAL, bool F16>
__global__ void __launch_bounds__(kBwdThreads, 1) fa_bwd_kernel(const __grid_constant__ BwdParams p) {
  using L = BwdLayout<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw;
  const uint32_t sbase = smem_u32(smem);
  // the 128-byte-swizzled tiles need 1024-byte alignment and there is no room for
  // padding: a misaligned window is reported, not used
  if ((sbase & 1023u) != 0) {
    if (threadIdx.x == 0) atomicCAS(&g_fa_status, 0ull, kStatusUnsupported);
    return;
  }
  // rejected sequence offsets (variable length): nothing to compute, nothing written
  if (p.cu_ok != nullptr && *p.cu_ok == 0) return;
  const uint32_t sK = sbase + L::kK, sV = sbase + L::kV, sQ = sbase + L::kQ, sDO = sbase + L::kDO,
                 sDS = sbase + L::kDS;
  auto bar = [&](int i) -> uint32_t { return sbase + L::kBar + 8u * (uint32_t)i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMisc + 4);
  volatile int* never_abort = reinterpret_cast<volatile int*>(smem + L::kMisc + 8);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  volatile int* task_slot = reinterpret_cast<volatile int*>(smem + L::kMisc + 16);   // [2]

  if (tid == 0) {
    *abort_flag = 0;
    *never_abort = 0;
    for (int i = 0; i < L::kNumBars; ++i) mbar_init(bar(i), 1);
    mbar_init(bar(L::bPReady), 256);
    mbar_init(bar(L::bdPEmpty), 128);
    mbar_init(bar(L::bdSReady), 256);
    mbar_init(bar(L::bdQStaged), 128);
    mbar_init(bar(L::bAccFree), 384);
    mbar_init(bar(L::bTaskEmpty + 0), L::kTaskReaders);
    mbar_init(bar(L::bTaskEmpty + 1), L::kTaskReaders);
    fence_mbar_init();
  }
  if (warp == 12 && lane == 0) {
    prefetch_tmap(&p.tm_q);
    prefetch_tmap(&p.tm_do);
    prefetch_tmap(&p.tm_k);
    prefetch_tmap(&p.tm_v);
  }
  if (warp == 8 && lane == 0) prefetch_tmap(&p.tm_dq);
  if (warp == 13) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // the tk-th task of this CTA as published by the producer warp (a whole warp calls
  // this; -1: give up). Readers free the slot once every lane has read it.
  auto next_task = [&](Waiter& w, int tk) -> int {
    if (!w.wait(bar(L::bTaskFull + (tk & 1)), (uint32_t)(tk >> 1) & 1u, L::bTaskFull + (tk & 1), tk)) return -1;
    const int idx = task_slot[tk & 1];
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(L::bTaskEmpty + (tk & 1)));
    return idx;
  };

  // register split 136 / 136 / 120 / 120 per thread for WG0 / WG1 / WG2 / WG3 (sum =
  // 4 x 128, the launch allocation)
  if (warp >= 12) {
    setmaxnreg_dec<120>();
    if (warp == 12) {
      // ============================================================ TMA producer
      Waiter w{abort_flag, p.timeout_ns, kRoleLoad};
      Tracer tr;
      tr.init(p.trace, p.trace_ctas, 0, lane == 0);
      const bool leader = elect_one();
      uint32_t q_armed = 0;   // bit s: stage s has an armed load whose completion may still be pending
      bool kv_armed = false;
      uint32_t q_par = 0;     // bit s: parity of the last arm of stage s
      uint32_t kv_par = 0;    // parity of the last arm of the K/V barrier
      bool ok = true;
      int g = 0;              // steps so far (all tasks of this CTA)
      int kvn = 0;            // tasks with steps so far
#pragma unroll 1
      for (int tk = 0; ok; ++tk) {
        // claim the next task and publish it
        if (!w.wait(bar(L::bTaskEmpty + (tk & 1)), ((uint32_t)(tk >> 1) & 1u) ^ 1u, L::bTaskEmpty + (tk & 1), tk)) {
          ok = false;
          break;
        }
        int ti = (int)blockIdx.x;
        if (tk > 0) ti = __shfl_sync(0xffffffffu, lane == 0 ? (int)gridDim.x + atomicAdd(p.task_counter, 1) : 0, 0);
        if (lane == 0) {
          task_slot[tk & 1] = ti;
          mbar_arrive(bar(L::bTaskFull + (tk & 1)));
        }
        __syncwarp();
        if (ti >= p.num_tasks) break;
        const BwdTask t = bwd_task<CAUSAL>(p, ti);
        if (t.n == 0) continue;
#pragma unroll 1
        for (int k = 0; k < t.n; ++k, ++g) {
          const int s = g & 1;
          const uint32_t use = (uint32_t)(g >> 1) & 1u;
          if (!w.wait(bar(L::bQEmpty + s), use ^ 1u, L::bQEmpty + s, g)) { ok = false; break; }
          const int i = t.i0 + k;
          const int tok = t.tok_q + ((i * 128) >> p.gshift);
          if (leader) {
            mbar_arrive_expect_tx(bar(L::bQFull + s), 2 * L::kTile + L::kStatsBytes);
#pragma unroll
            for (int c = 0; c < L::kHalves; ++c) {
              tma_load_3d(sQ + s * L::kTile + c * L::kSlab, &p.tm_q, c * 64, t.kvh << p.gshift, tok,
                          bar(L::bQFull + s));
              tma_load_3d(sDO + s * L::kTile + c * L::kSlab, &p.tm_do, c * 64, t.kvh << p.gshift, tok,
                          bar(L::bQFull + s));
            }
            const size_t pk = ((size_t)t.b * p.Hkv + t.kvh) * p.mpad + (size_t)i * 128;
            const uint32_t st = sbase + L::kStats + s * L::kStatsBytes;
            bulk_load(st, p.lse2 + pk, 512, bar(L::bQFull + s));
            bulk_load(st + 512, p.dsum + pk, 512, bar(L::bQFull + s));
          }
          __syncwarp();
          tr.rec(kEvBQLoad, g);
          q_armed |= 1u << s;
          q_par = (q_par & ~(1u << s)) | (use << s);
          if (k == 0) {
            // this task's K and V, once the previous task's products have read theirs
            if (kvn > 0 && !w.wait(bar(L::bFinal), (uint32_t)(kvn - 1) & 1u, L::bFinal, g)) { ok = false; break; }
            if (leader) {
              mbar_arrive_expect_tx(bar(L::bKV), 2 * L::kTile);
#pragma unroll
              for (int c = 0; c < L::kHalves; ++c) {
                tma_load_3d(sK + c * L::kSlab, &p.tm_k, c * 64, t.kvh, t.tok_k + t.j * 128, bar(L::bKV));
                tma_load_3d(sV + c * L::kSlab, &p.tm_v, c * 64, t.kvh, t.tok_k + t.j * 128, bar(L::bKV));
              }
            }
            __syncwarp();
            kv_armed = true;
            kv_par = (uint32_t)kvn & 1u;
            ++kvn;
          }
        }
      }
      if (!ok) {
        Waiter d{never_abort, p.timeout_ns, kRoleDrain};
        if (kv_armed) d.wait(bar(L::bKV), kv_par, L::bKV, -1);
#pragma unroll 1
        for (int s = 0; s < 2; ++s)
          if (q_armed & (1u << s)) d.wait(bar(L::bQFull + s), (q_par >> s) & 1, L::bQFull + s, -1);
      }
    } else if (warp == 13) {
      // ============================================================ MMA issuer
      Waiter w{abort_flag, p.timeout_ns, kRoleMma};
      Tracer tr;
      tr.init(p.trace, p.trace_ctas, 1, lane == 0);
      const bool leader = elect_one();
      constexpr uint32_t idS = idesc_f32acc2(128, 128, false, false, F16);   // S^T, dP^T: both K-major
      constexpr uint32_t idV = idesc_f32acc2(128, D, false, true, F16);      // dV: A = P^T (TMEM), B = dO MN-major
      constexpr uint32_t idK = idesc_f32acc2(128, D, false, true, F16);      // dK: A = dS^T K-major, B = Q MN-major
      constexpr uint32_t idQ = idesc_f32acc2(128, D, true, true, F16);       // dQ: A = dS MN-major, B = K MN-major
      const uint64_t Kk = smem_desc_sw128(sK, 16, 1024), Vk = smem_desc_sw128(sV, 16, 1024);
      const uint64_t Kmn = smem_desc_sw128(sK, L::kSlab, 1024);
      const uint64_t dSk = smem_desc_sw128(sDS, 16, 1024), dSmn = smem_desc_sw128(sDS, L::kSlab, 1024);
      const uint32_t tS = tmem + L::cS, tP = tmem + L::cS + 32, tdP = tmem + L::cDP;
      const uint32_t tdV = tmem + L::cDV, tdK = tmem + L::cDK;
      auto qk = [&](int s) { return smem_desc_sw128(sQ + s * L::kTile, 16, 1024); };
      auto qmn = [&](int s) { return smem_desc_sw128(sQ + s * L::kTile, L::kSlab, 1024); };
      auto dok = [&](int s) { return smem_desc_sw128(sDO + s * L::kTile, 16, 1024); };
      auto domn = [&](int s) { return smem_desc_sw128(sDO + s * L::kTile, L::kSlab, 1024); };
      // S^T = K Q_s^T (M = keys, N = rows, K = d)
      auto issue_s = [&](int s) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t o = kmajor_step<L::kSlab>(kk) >> 4;
          mma_ss(tS, Kk + o, qk(s) + o, idS, kk > 0 ? 1u : 0u);
        }
      };
      // dP^T = V dO_s^T
      auto issue_dp = [&](int s) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t o = kmajor_step<L::kSlab>(kk) >> 4;
          mma_ss(tdP, Vk + o, dok(s) + o, idS, kk > 0 ? 1u : 0u);
        }
      };
      bool ok = true;
      int g = 0, kvn = 0;
#pragma unroll 1
      for (int tk = 0; ok; ++tk) {
        const int ti = next_task(w, tk);
        if (ti < 0) {
          ok = false;
          break;
        }
        if (ti >= p.num_tasks) break;
        const BwdTask t = bwd_task<CAUSAL>(p, ti);
        const int n = t.n;
        if (n == 0) continue;
        // prologue: S^T and dP^T of the first tile, once K, V and its Q, dO have landed
        // (dP^T also once WG2 has taken the previous task's last dQ out of its columns)
        ok = w.wait(bar(L::bKV), (uint32_t)kvn & 1u, L::bKV, g);
        if (ok) ok = w.wait(bar(L::bQFull + (g & 1)), (uint32_t)(g >> 1) & 1u, L::bQFull + (g & 1), g);
        if (ok) {
          tc_fence_after();
          if (leader) {
            issue_s(g & 1);
            mma_commit(bar(L::bSFull));
          }
          __syncwarp();
          ok = w.wait(bar(L::bdPEmpty), (uint32_t)g & 1u, L::bdPEmpty, g);
        }
        if (ok) {
          tc_fence_after();
          if (leader) {
            issue_dp(g & 1);
            mma_commit(bar(L::bdPFull));
          }
          __syncwarp();
        }
#pragma unroll 1
        for (int k = 0; ok && k < n; ++k) {
          const int gg = g + k;
          const int s = gg & 1;
          // dV += P^T dO (K = 128 rows: P^T from TMEM, 8 columns of 16-bit pairs per step;
          // rows 0-63 in columns [32, 64) of S^T, rows 64-127 in [96, 128)); the first
          // step overwrites dV (and dK below) once the previous task's write-out has read them
          if (!w.wait(bar(L::bPReady), (uint32_t)gg & 1u, L::bPReady, gg)) { ok = false; break; }
          if (k == 0 && kvn > 0 &&
              !w.wait(bar(L::bAccFree), (uint32_t)(kvn - 1) & 1u, L::bAccFree, gg)) { ok = false; break; }
          tc_fence_after();
          if (leader) {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_ts(tdV, tP + (kk >> 2) * 64 + (kk & 3) * 8, domn(s) + ((kk * 2048) >> 4), idV,
                     (k > 0 || kk > 0) ? 1u : 0u);
          }
          __syncwarp();
          tr.rec(kEvBdV, gg);
          // dK += dS^T Q and dQ = dS K (once dS is in shared memory) and the next tile's
          // S^T (once its Q has landed; its columns are free, the dV above has read P^T):
          // whichever input arrives first is issued first (non-blocking tests: a try_wait
          // on the barrier that is not ready would hold the warp until that one completes)
          {
            const int s1 = (gg + 1) & 1;
            bool s_done = k + 1 >= n, dq_done = false;
            uint32_t it = 0;
            uint64_t t0 = 0;
            while (!(s_done && dq_done)) {
              if (!s_done &&
                  __all_sync(0xffffffffu, mbar_test_wait(bar(L::bQFull + s1), (uint32_t)((gg + 1) >> 1) & 1u))) {
                tc_fence_after();
                if (leader) {
                  issue_s(s1);
                  mma_commit(bar(L::bSFull));
                }
                __syncwarp();
                tr.rec(kEvBS, gg + 1);
                s_done = true;
                continue;
              }
              if (!dq_done && __all_sync(0xffffffffu, mbar_test_wait(bar(L::bdSReady), (uint32_t)gg & 1u))) {
                tc_fence_after();
                if (leader) {
                  // dQ first, so WG2 can start on it while dK runs
#pragma unroll
                  for (int kk = 0; kk < 8; ++kk)
                    mma_ss(tdP, dSmn + ((kk * 2048) >> 4), Kmn + ((kk * 2048) >> 4), idQ, kk > 0 ? 1u : 0u);
                  mma_commit(bar(L::bdQFull));
#pragma unroll
                  for (int kk = 0; kk < 8; ++kk)
                    mma_ss(tdK, dSk + (kmajor_step<L::kSlab>(kk) >> 4), qmn(s) + ((kk * 2048) >> 4), idK,
                           (k > 0 || kk > 0) ? 1u : 0u);
                  mma_commit(bar(L::bdSEmpty));  // also: this step's Q and dO are no longer read
                }
                __syncwarp();
                tr.rec(kEvBdKdQ, gg);
                dq_done = true;
                continue;
              }
              if (!w.still_waiting(it, t0, dq_done ? L::bQFull + s1 : L::bdSReady, gg)) { ok = false; break; }
            }
            if (!ok) break;
          }
          // the next tile's dP^T, once WG2 has taken dQ out of those columns
          if (k + 1 < n) {
            const int s1 = (gg + 1) & 1;
            if (!w.wait(bar(L::bdPEmpty), (uint32_t)(gg + 1) & 1u, L::bdPEmpty, gg + 1)) { ok = false; break; }
            tc_fence_after();
            if (leader) {
              issue_dp(s1);
              mma_commit(bar(L::bdPFull));
            }
            __syncwarp();
            tr.rec(kEvBdP, gg + 1);
          }
        }
        if (ok && leader) mma_commit(bar(L::bFinal));   // this task's products are done (K, V, dK, dV)
        __syncwarp();
        g += n;
        ++kvn;
      }
      // every issued MMA must finish before the tensor memory is released
      if (leader) mma_commit(bar(L::bDrain));
      __syncwarp();
      Waiter d{never_abort, p.timeout_ns, kRoleDrain};
      d.wait(bar(L::bDrain), 0, L::bDrain, -1);
    }
  } else if (warp < 8) {
    // ================================================================ WG0 / WG1: P and dS (one key per thread)
    setmaxnreg_inc<136>();
    const int hq = warp >> 2;                             // query columns [64 hq, 64 hq + 64) of the tile
    const int cq = hq * 64;
    const int kr = tid & 127;                             // key row == TMEM lane
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_base + L::cS + cq, tdP = tmem + lane_base + L::cDP + cq;
    Waiter w{abort_flag, p.timeout_ns, hq == 0 ? kRoleSoftmax0 : kRoleSoftmax1};
    Tracer tr;
    tr.init(p.trace, p.trace_ctas, 2 + hq, kr == 0);
    const float sl2 = p.scale_log2, sc = p.scale;
    bool ok = true;
    int g = 0, kvn = 0;
#pragma unroll 1
    for (int tk = 0; ok; ++tk) {
      const int ti = next_task(w, tk);
      if (ti < 0) {
        ok = false;
        break;
      }
      if (ti >= p.num_tasks) break;
      const BwdTask t = bwd_task<CAUSAL>(p, ti);
      if (t.skip) continue;
      const int n = t.n;
      const int kabs = t.j * 128 + kr;
      const bool key_ok = kabs < t.Nk;
#pragma unroll 1
      for (int k = 0; k < n; ++k) {
        const int gg = g + k;
        const int i = t.i0 + k;
        // this tile's base-2 LSE and D, loaded with Q and dO (q_full of the stage, waited below)
        const float4* L2 = reinterpret_cast<const float4*>(smem + L::kStats + (gg & 1) * L::kStatsBytes) + cq / 4;
        const float4* DS = L2 + 32;
        // rows [qlo, qhi) of this tile see this key: causal needs position >= kabs - off,
        // and rows past the sequence's packed end are padding (local to this half)
        const int qlo = CAUSAL ? (int)max(-1LL, min(129LL, ((long long)kabs - t.off) * (1LL << p.gshift) -
                                                               (long long)i * 128)) - cq
                               : -cq;
        const int qhi = (key_ok ? min(128, (t.Nq << p.gshift) - i * 128) : 0) - cq;
        if (!w.wait(bar(L::bQFull + (gg & 1)), (uint32_t)(gg >> 1) & 1u, L::bQFull + (gg & 1), gg)) { ok = false; break; }
        if (!w.wait(bar(L::bSFull), (uint32_t)gg & 1u, L::bSFull, gg)) { ok = false; break; }
        tr.rec(kEvBSFull, gg);
        tc_fence_after();
        float P[64];
        {
          uint32_t u[64];
          tmem_ld32(tS, *reinterpret_cast<uint32_t(*)[32]>(&u[0]));
          tmem_ld32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&u[32]));
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < 64; c += 4) {
            const float4 l = L2[c / 4];
            const float lv[4] = {l.x, l.y, l.z, l.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int q = c + e;
              const float x = fmaf(__uint_as_float(u[q]), sl2, -lv[e]);
              P[q] = (q >= qlo && q < qhi) ? ex2_approx(x) : 0.f;
            }
          }
        }
        // P^T as 16-bit pairs over the upper 32 columns of this half of S^T (all of the
        // half was read above): the A operand of dV
        {
          uint32_t pk[32];
#pragma unroll
          for (int c = 0; c < 32; ++c) pk[c] = pack_16x2<F16>(P[2 * c], P[2 * c + 1]);
          tmem_st32(tS + 32, pk);
          tmem_wait_st();
        }
        tc_fence_before();
        mbar_arrive(bar(L::bPReady));
        tr.rec(kEvBPReady, gg);
        // dS = s * P * (dP - D) -> 16-bit -> slab hq of the shared dS tile (row = key, 128-byte
        // swizzle), stored once the previous step's dK has finished reading the tile
        if (!w.wait(bar(L::bdPFull), (uint32_t)gg & 1u, L::bdPFull, gg)) { ok = false; break; }
        tr.rec(kEvBdPFull, gg);
        tc_fence_after();
        uint32_t pk[32];
#pragma unroll
        for (int ch = 0; ch < 2; ++ch) {
          uint32_t u[32];
          tmem_ld32(tdP + ch * 32, u);
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < 32; c += 4) {
            const float4 dd = DS[(ch * 32 + c) / 4];
            const float dv[4] = {dd.x, dd.y, dd.z, dd.w};
            float gr[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) gr[e] = P[ch * 32 + c + e] * (__uint_as_float(u[c + e]) - dv[e]) * sc;
            pk[(ch * 32 + c) / 2] = pack_16x2<F16>(gr[0], gr[1]);
            pk[(ch * 32 + c) / 2 + 1] = pack_16x2<F16>(gr[2], gr[3]);
          }
        }
        if (gg > 0 && !w.wait(bar(L::bdSEmpty), (uint32_t)(gg - 1) & 1u, L::bdSEmpty, gg)) { ok = false; break; }
        const uint32_t row = sDS + (uint32_t)hq * L::kSlab + (uint32_t)kr * 128u;
#pragma unroll
        for (int uu = 0; uu < 8; ++uu)
          st_shared_v4(row + (((uint32_t)uu ^ (uint32_t)(kr & 7)) << 4), pk[4 * uu], pk[4 * uu + 1], pk[4 * uu + 2],
                       pk[4 * uu + 3]);
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(bar(L::bdSReady));
        tr.rec(kEvBdSReady, gg);
      }
      if (!ok) break;
      // dK (scale already in dS) -> 16-bit -> global; this warpgroup writes columns
      // [hq * D / 2, (hq + 1) * D / 2). Its tensor-memory columns are read first, then
      // handed back (b_acc_free) before the stores.
      if (n > 0 && !w.wait(bar(L::bFinal), (uint32_t)kvn & 1u, L::bFinal, -1)) { ok = false; break; }
      if (n > 0) tc_fence_after();
      uint16_t* dst = p.dk + ((size_t)(t.tok_k + kabs) * p.Hkv + t.kvh) * D;
#pragma unroll 1
      for (int c = hq * (D / 64); c < (hq + 1) * (D / 64); ++c) {
        uint32_t u[32];
        if (n > 0) {
          tmem_ld32(tmem + lane_base + L::cDK + c * 32, u);
          tmem_wait_ld();
          if (c == (hq + 1) * (D / 64) - 1) {   // the last read of this warpgroup's columns
            tc_fence_before();
            mbar_arrive(bar(L::bAccFree));
          }
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) u[e] = 0u;
        }
        if (key_ok) {
          uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
          for (int e = 0; e < 4; ++e)
            d4[e] = make_uint4(pack_16x2<F16>(__uint_as_float(u[8 * e]), __uint_as_float(u[8 * e + 1])),
                               pack_16x2<F16>(__uint_as_float(u[8 * e + 2]), __uint_as_float(u[8 * e + 3])),
                               pack_16x2<F16>(__uint_as_float(u[8 * e + 4]), __uint_as_float(u[8 * e + 5])),
                               pack_16x2<F16>(__uint_as_float(u[8 * e + 6]), __uint_as_float(u[8 * e + 7])));
        }
      }
      if (n > 0) {
        g += n;
        ++kvn;
      }
    }
  } else if (warp < 12) {
    // ================================================================ WG2: dQ reduce-adds, then dV
    setmaxnreg_dec<120>();
    const int r = tid - 256;                              // Q-tile row (dQ) / key row (dV) == TMEM lane
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    Waiter w{abort_flag, p.timeout_ns, kRoleCorr};
    Tracer tr;
    tr.init(p.trace, p.trace_ctas, 4, r == 0);
    mbar_arrive(bar(L::bdPEmpty));                        // the dP columns start free
    bool ok = true;
    int g = 0, kvn = 0;
#pragma unroll 1
    for (int tk = 0; ok; ++tk) {
      const int ti = next_task(w, tk);
      if (ti < 0) {
        ok = false;
        break;
      }
      if (ti >= p.num_tasks) break;
      const BwdTask t = bwd_task<CAUSAL>(p, ti);
      if (t.skip) continue;
      const int n = t.n;
#pragma unroll 1
      for (int k = 0; k < n; ++k) {
        const int gg = g + k;
        const int i = t.i0 + k;
        const int s = gg & 1;
        const bool valid = ((i * 128 + r) >> p.gshift) < t.Nq;   // padding rows add zeros
        if (!w.wait(bar(L::bdQFull), (uint32_t)gg & 1u, L::bdQFull, gg)) { ok = false; break; }
        tr.rec(kEvBdQFull, gg);
        tc_fence_after();
        // dQ in 32-column chunks -> fp32 rows in the freed dO_s / Q_s buffers, in the
        // 128-byte-swizzled layout of the reduce map (16-byte unit u of row r at u ^ (r % 8)).
        // dO_s is free once dQ is done (dV and dP, the products that read it, came before);
        // Q_s only once dK (issued after dQ) is done: round 0 stages the upper chunks in
        // dO_s, round 1 loads the lower chunks, frees the TMEM columns, waits for dK and
        // stages them in Q_s. Each round's reduce-adds leave once all 128 rows are staged.
        const int tok = t.tok_q + ((i * 128) >> p.gshift);
        auto stage_chunk = [&](const uint32_t (&u)[32], uint32_t chunk) {
          const uint32_t row = chunk + (uint32_t)r * 128u;
#pragma unroll
          for (int uu = 0; uu < 8; ++uu) {
            const uint32_t a0 = valid ? u[4 * uu] : 0u, a1 = valid ? u[4 * uu + 1] : 0u;
            const uint32_t a2 = valid ? u[4 * uu + 2] : 0u, a3 = valid ? u[4 * uu + 3] : 0u;
            st_shared_v4(row + (((uint32_t)uu ^ (uint32_t)(r & 7)) << 4), a0, a1, a2, a3);
          }
        };
        int* sem = p.sem != nullptr ? p.sem + ((size_t)t.b * p.Hkv + t.kvh) * p.ntiles + i : nullptr;
        // All rows of the round staged: send them. Every warp waits for the round's phase,
        // so that none arrives for the next round before this phase has completed (warp 8
        // may be held below, waiting for its turn).
        // Deterministic order: the key blocks add this tile's dQ one after another (key
        // block j once blocks 0 .. j-1 have), so warp 8 sends both rounds together in
        // round 1, after a bounded wait for its turn. The wait comes after this tile's
        // bdSEmpty has been observed: while warp 8 waits, the MMA warp may complete the
        // next tile's dK, and a parity wait on bdSEmpty two phases behind would never end.
        auto send = [&](int rnd) {
          if (lane == 0) {
#pragma unroll
            for (int h = 0; h < L::kHalves; ++h) {
              const int c = rnd == 0 ? L::kHalves + h : h;
              const uint32_t chunk = (rnd == 0 ? sDO : sQ) + s * L::kTile + h * L::kSlab;
              tma_reduce_add_3d(&p.tm_dq, chunk, c * 32, t.kvh << p.gshift, tok);
            }
          }
        };
        auto round_done = [&](int rnd) -> bool {
          fence_proxy_async_smem();
          mbar_arrive(bar(L::bdQStaged));
          if (!w.wait(bar(L::bdQStaged), (uint32_t)rnd, L::bdQStaged, gg)) return false;
          if (warp == 8) {
            if (sem == nullptr) {
              send(rnd);
            } else if (rnd == 1) {
              uint32_t it = 0;
              uint64_t t0 = 0;
              while (__shfl_sync(0xffffffffu, lane == 0 ? ld_acquire_gpu(sem) : 0, 0) != t.j)
                if (!w.still_waiting(it, t0, L::kNumBars, gg)) return false;
              fence_proxy_async_global();
              send(0);
              send(1);
            }
            __syncwarp();
          }
          return true;
        };
#pragma unroll 1
        for (int h = 0; h < L::kHalves; ++h) {
          uint32_t u[32];
          tmem_ld32(tmem + lane_base + L::cDP + (L::kHalves + h) * 32, u);
          tmem_wait_ld();
          stage_chunk(u, sDO + s * L::kTile + h * L::kSlab);
        }
        {
          uint32_t u[L::kHalves][32];
#pragma unroll
          for (int h = 0; h < L::kHalves; ++h) tmem_ld32(tmem + lane_base + L::cDP + h * 32, u[h]);
          tmem_wait_ld();
          tc_fence_before();
          mbar_arrive(bar(L::bdPEmpty));                  // all of dQ has left TMEM: free the columns
          tr.rec(kEvBdPEmpty, gg);
          if (!round_done(0)) { ok = false; break; }
          if (!w.wait(bar(L::bdSEmpty), (uint32_t)gg & 1u, L::bdSEmpty, gg)) { ok = false; break; }   // dK has read Q_s
#pragma unroll
          for (int h = 0; h < L::kHalves; ++h) stage_chunk(u[h], sQ + s * L::kTile + h * L::kSlab);
        }
        if (!round_done(1)) { ok = false; break; }
        tr.rec(kEvBStaged, gg);
        if (warp == 8) {
          if (lane == 0) {
            bulk_commit();
            if (sem != nullptr) {
              bulk_wait_all();                            // the additions are done: pass the turn on
              fence_proxy_async_global();
              st_release_gpu(sem, t.j + 1);
            } else {
              bulk_wait_read_all();                       // the staging may be overwritten now
            }
            mbar_arrive(bar(L::bQEmpty + s));             // Q_s and dO_s may be reloaded
            tr.rec(kEvBReduced, gg);
          }
          __syncwarp();
        }
      }
      if (!ok) break;
      // dV -> 16-bit -> global: all of its tensor-memory columns are read (b_acc_free
      // follows the last read), then stored
      if (n > 0 && !w.wait(bar(L::bFinal), (uint32_t)kvn & 1u, L::bFinal, -1)) { ok = false; break; }
      const int kabs = t.j * 128 + r;
      uint16_t* dst = p.dv + ((size_t)(t.tok_k + kabs) * p.Hkv + t.kvh) * D;
      if (n > 0) tc_fence_after();
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t u[32];
        if (n > 0) {
          tmem_ld32(tmem + lane_base + L::cDV + c * 32, u);
          tmem_wait_ld();
          if (c == D / 32 - 1) {
            tc_fence_before();
            mbar_arrive(bar(L::bAccFree));
          }
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) u[e] = 0u;
        }
        if (kabs < t.Nk) {
          uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
          for (int e = 0; e < 4; ++e)
            d4[e] = make_uint4(pack_16x2<F16>(__uint_as_float(u[8 * e]), __uint_as_float(u[8 * e + 1])),
                               pack_16x2<F16>(__uint_as_float(u[8 * e + 2]), __uint_as_float(u[8 * e + 3])),
                               pack_16x2<F16>(__uint_as_float(u[8 * e + 4]), __uint_as_float(u[8 * e + 5])),
                               pack_16x2<F16>(__uint_as_float(u[8 * e + 6]), __uint_as_float(u[8 * e + 7])));
        }
      }
      if (n > 0) {
        g += n;
        ++kvn;
      }
    }
    if (warp == 8 && lane == 0) bulk_wait_all();          // reduce-adds complete before exit
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 13) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace fa
