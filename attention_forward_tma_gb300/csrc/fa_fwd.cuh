// fa_fwd.cuh -- the attention forward kernel for GB300 (sm_103a).
//
// One CTA of 512 threads works on tasks of 256 query rows of one (sequence,
// K/V head): two Q tiles of 128 rows that share every streamed K/V block. With
// grouped-query attention (G = H / H_kv query heads per K/V head, G a power of
// two up to 128) the rows of a tile are packed: row r holds sequence position
// tile_pos0 + r / G of query head kv * G + r % G, so one K/V block serves all
// G heads ("Flash Attention 4", section "GQA 支持"); G = 1 is plain multi-head
// attention. The four warpgroups have fixed roles ("Flash Attention 4", section
// "Warp 角色与 Scope"):
//
//   WG0, WG1  softmax of Q tile 0 / Q tile 1 (thread r owns row r of its tile)
//   WG2       correction (rescale of O in tensor memory) and the epilogue
//             (O / row_sum -> bf16 or fp16 -> global memory)
//   WG3       warp 12: tcgen05 MMA issue; warp 13: TMA loads and task claims
//             (work stealing by cluster launch control); warps 14-15 idle
//
// Per K/V block j (visited from the last block down to block 0, section
// "Pipeline 时间线"):   S_t = Q_t K_j^T  (tcgen05, smem x smem -> TMEM fp32)
//                      P_t = exp2(S_t * scale_log2 - ref_t * scale_log2)  (registers,
//                            written back to TMEM as bf16 / fp16 (the input type)
//                            over the upper half of S_t)
//                      O_t (+)= P_t V_j  (tcgen05, A from TMEM, B from smem)
// with the delayed-rescale rule of section "算法结构": the reference ref_t of a
// row moves to the new maximum only when that maximum exceeds it by more than
// tau (base-2 exponent units); then O and row_sum are multiplied by
// acc_scale = 2^delta. The rescale of O is done by WG2, which skips a warp's 32
// rows when none of them needs it (section "重缩放与结果写回").
//
// Tensor memory (512 columns x 128 lanes x 32 bit, section "TMEM 布局与复用"):
//   S_0 [0,128)   S_1 [128,256)   O_0 [256,256+D)   O_1 [384,384+D)
//   P_t = 16-bit (bf16 / fp16) pairs over columns [64,128) of S_t.
//
// Shared memory: Q tiles (2), a ring of K/V stages (K and V blocks alternate
// through the same ring), the O staging tile of the TMA store, mbarriers, and a
// 2x128 float mailbox that carries each row's final row_sum from the softmax
// warpgroups to WG2 (acc_scale goes through column 0 of S_t, or through the
// mailbox when the statistics option selects shared memory).
//
// Every wait is bounded: after FwdParams::timeout_ns a waiter records
// FA_ERR_TIMEOUT in g_fa_status, raises a CTA-wide abort flag and unwinds;
// the CTA then drains its own TMA copies and MMAs (again with a bound), frees
// its tensor memory and exits.
#pragma once

#include <cstdint>

#include "ptx.cuh"

#ifndef FA_KV_STAGES_D128
#define FA_KV_STAGES_D128 4
#endif

namespace fa {

constexpr int kBlockM = 128;          // rows of one Q tile
constexpr int kBlockN = 128;          // keys of one K/V block
constexpr int kTaskRows = 2 * kBlockM;
constexpr int kSplitP = 96;           // two-tile tasks hand P to the PV MMA as keys [0, 96) and [96, 128)
constexpr int kSoloSplitP = 64;       // solo tasks: one half per softmax warpgroup
constexpr int kThreads = 512;
constexpr uint32_t kTmemCols = 512;

// Device status word: 0 = OK; else code | role << 8 | barrier << 16 | block << 32.
static __device__ unsigned long long g_fa_status;  // one copy per translation unit

enum : uint32_t { kRoleMma = 1, kRoleLoad = 2, kRoleSoftmax0 = 3, kRoleSoftmax1 = 4, kRoleCorr = 5,
                  kRoleDrain = 6 };
constexpr unsigned long long kStatusTimeout = 4;  // == FA_ERR_TIMEOUT
constexpr unsigned long long kStatusUnsupported = 2;  // == FA_ERR_UNSUPPORTED

struct FwdParams {
  // 3-D maps of [tokens, heads, d]: x = d, y = head, z = token. Q and O: box
  // 64 x G x 128/G (one packed 128-row tile); K and V: box 64 x 1 x 128.
  CUtensorMap tm_q, tm_k, tm_v;
  CUtensorMap tm_o;              // the view of O for the TMA store of full tiles
  uint16_t* o;                   // [tokens, H, d] bf16 / fp16 (splits == 1)
  float* lse;                    // fixed length [B, H, N]; varlen [H, tokens]; may be null (splits == 1)
  // splits > 1: the keys of every task are cut into `splits` ranges of whole
  // blocks, computed as separate tasks; each writes its normalised fp32 O and its
  // LSE (-inf: no key in the range) here, and a merge kernel combines them.
  float* o_part;                 // [splits, tokens, H, d]
  float* lse_part;               // [splits, LSE layout]
  long long lse_split_stride;    // elements between the splits of lse_part
  int splits;
  int part_out;                  // 1: write o_part / lse_part (splits > 1, or one key shard of a longer
                                 // sequence whose partial result another call or device merges)
  int pdl;                       // 1: launched with programmatic stream serialization
  int diag_shift;                // fixed length: keys of the sequence after the last key given (a key
                                 // shard's causal diagonal stays the full sequence's); else 0
  const int* cu_seqlens;         // varlen only: query rows of each sequence
  const int* cu_seqlens_k;       // varlen only: key rows of each sequence
  const int4* tasks;             // varlen only: {seq, kv head | split << 16, m_block, cost}, longest first
  const int* task_count;         // varlen only
  int B, H, N;                   // fixed length: batch, query heads, query rows per sequence
  int Nk;                        // fixed length: key rows per sequence
  int Hkv;                       // K/V heads; H = Hkv << gshift
  int gshift;                    // log2 of G, the query heads per K/V head (packed rows per position)
  int total_tokens;              // rows of Q and O
  int num_tasks;                 // fixed length: exact; varlen: upper bound (grid sizing)
  int num_m;                     // fixed length: task_rows-row blocks of packed rows per (b, kv head)
  int task_rows;                 // packed rows per task: 256 (two Q tiles) or 128 (solo: one Q tile whose
                                 // score tile alternates between S_0 and S_1)
  int lpt_group;                 // causal fixed length: (b, kv head) pairs per L2 section
  int varlen;
  float scale_log2;              // scale * log2(e)
  float tau;                     // delayed-rescale threshold
  int emu_groups;                // 16-column groups per row evaluated with the polynomial exp2
  int sched;                     // 0: one task per CTA; 1: static stride; 2: work stealing (launch control)
  int stagger;                   // 1: WG0 and WG1 take turns at their exponential phases
  int stats_tmem;                // 1: acc_scale goes to WG2 through tensor memory (column 0 of S_t)
  unsigned long long timeout_ns;
  unsigned long long* trace;     // tracing build only: clock stamps per CTA and role (else null)
  int trace_ctas;
};

// ------------------------------------------------------------------ tracing (FA_TRACE builds)
// A tracing build stamps the SM clock at every hand-off of the pipeline for the
// first trace_ctas CTAs: one leader thread per role writes one 64-bit word per
// event, (32-bit clock << 32) | (event code << 24) | (block & 0xffffff), into
// trace[(cta * kTraceRoles + role) * kTraceSlots + n]; the buffer starts zeroed,
// so the first zero word ends a role's events. One clock read and one store per
// event keep the stamps' own cost small. Normal builds compile the stamps away.
constexpr int kTraceRoles = 5;      // producer, MMA, softmax 0, softmax 1, correction
constexpr int kTraceSlots = 8192;   // 64-bit words (events) per role
enum : uint32_t {
  kEvQ0 = 1, kEvK = 2, kEvQ1 = 3, kEvV = 4,
  kEvS0 = 10, kEvS1 = 11, kEvPO0 = 12, kEvPV0a = 13, kEvP20 = 14, kEvPV0b = 15, kEvPO1 = 16,
  kEvPV1a = 17, kEvP21 = 18, kEvPV1b = 19, kEvKVV = 20, kEvKVK = 21,
  kEvSFull = 30, kEvSMax = 31, kEvMail = 32, kEvHalf1 = 33, kEvHalf2 = 34, kEvStats = 35,
  kEvCorrFull = 40, kEvCorrDone = 42, kEvEpiStart = 44, kEvEpiEnd = 46, kEvTask = 48,
  kEvIssueBegin = 50,
  // backward: producer, MMA issuer, P/dS warpgroups (roles 2, 3), dQ warpgroup (role 4)
  kEvBQLoad = 60, kEvBdV = 61, kEvBS = 62, kEvBdKdQ = 63, kEvBdP = 64, kEvBSFull = 70, kEvBPReady = 71,
  kEvBdPFull = 72, kEvBdSReady = 73, kEvBdQFull = 80, kEvBdPEmpty = 81, kEvBStaged = 82, kEvBReduced = 83
};
struct Tracer {
#ifdef FA_TRACE
  unsigned long long* buf = nullptr;
  uint32_t n = 0;
  __device__ __forceinline__ void init(unsigned long long* trace, int trace_ctas, int role, bool leader) {
    if (leader && trace != nullptr && (int)blockIdx.x < trace_ctas)
      buf = trace + ((size_t)blockIdx.x * kTraceRoles + role) * kTraceSlots;
  }
  __device__ __forceinline__ void init(const FwdParams& p, int role, bool leader) {
    init(p.trace, p.trace_ctas, role, leader);
  }
  __device__ __forceinline__ void rec(uint32_t code, int blk) {
    if (buf != nullptr && n < (uint32_t)kTraceSlots) {
      uint32_t c;
      asm volatile("mov.u32 %0, %%clock;" : "=r"(c));
      buf[n++] = ((unsigned long long)c << 32) | (code << 24) | ((uint32_t)blk & 0xffffffu);
    }
  }
#else
  __device__ __forceinline__ void init(unsigned long long*, int, int, bool) {}
  __device__ __forceinline__ void init(const FwdParams&, int, bool) {}
  __device__ __forceinline__ void rec(uint32_t, int) {}
#endif
};

template <int D>
struct Layout {
  static_assert(D == 64 || D == 128, "head dim");
  static constexpr int kHalves = D / 64;                   // 128-byte (64-element) column slabs
  static constexpr int kSlabBytes = kBlockM * 128;          // one slab: 128 rows x 128 bytes
  static constexpr int kTileBytes = kHalves * kSlabBytes;   // one Q, K or V tile
  static constexpr int kStages = D == 128 ? FA_KV_STAGES_D128 : 8;  // K/V ring depth
  static constexpr int kQOff = 0;
  static constexpr int kKVOff = kQOff + 2 * kTileBytes;
  static constexpr int kOstOff = kKVOff + kStages * kTileBytes;  // O staging tile for the TMA store
  static constexpr int kBarOff = kOstOff + kTileBytes;
  // barrier indices
  static constexpr int bQFull = 0, bQEmpty = 2, bKVFull = 4, bKVEmpty = 4 + kStages;
  static constexpr int bSFull = 4 + 2 * kStages, bPO = bSFull + 2, bP2 = bPO + 2, bCorrFull = bP2 + 2,
                       bCorrEmpty = bCorrFull + 2, bOFinal = bCorrEmpty + 2, bDrain = bOFinal + 2,
                       bTaskFull = bDrain + 1, bTaskEmpty = bTaskFull + 2, bClc = bTaskEmpty + 2,
                       bOstReady = bClc + 1, bOstFree = bOstReady + 1, bTurn = bOstFree + 1,
                       bStats = bTurn + 2, bPVDone = bStats + 2, bXchg = bPVDone + 1, bRowSum = bXchg + 2;
  static constexpr int kNumBars = bRowSum + 1;
  static constexpr int kMailOff = kBarOff + ((kNumBars * 8 + 127) / 128) * 128;
  static constexpr int kMiscOff = kMailOff + 2 * kBlockM * 4;  // tmem slot, abort flags, task ring
  static constexpr int kClcOff = kMiscOff + 64;                 // 16-byte launch-control response
  static constexpr int kSmemBytes = kClcOff + 16;
  static constexpr int kSmemAlloc = kSmemBytes + 1024;         // slack for 1024-byte alignment
  static_assert(kSmemAlloc <= 227 * 1024, "shared memory per CTA");
  // tensor memory columns of S_t and O_t
  static __device__ __forceinline__ uint32_t col_s(int t) { return (uint32_t)t * 128u; }
  static __device__ __forceinline__ uint32_t col_o(int t) { return 256u + (uint32_t)t * 128u; }
};

// ------------------------------------------------------------------ tasks
struct Task {
  int kvh, tok0, len;      // K/V head, first query row of the sequence, its length
  int row0, rows;          // the task's packed rows [row0, row0 + rows) of the sequence (rows 256 or 128)
  int tok0k, lenk;         // first key row of the sequence, its number of keys
  int off;                 // causal offset: position i sees keys j <= i + off
  int split;               // key range (splits > 1)
  int lse_base;            // lse index of position 0 of query head kvh * G
  int lse_hstride;         // lse distance between consecutive query heads
};

// First sequence position of the packed rows from `row` on (row a multiple of G).
__device__ __forceinline__ int packed_pos(const Task& t, int row, int gshift) {
  return (t.row0 + row) >> gshift;
}

// ROWS: packed rows per task (256, or 128 in a solo kernel).
template <int ROWS>
__device__ __forceinline__ bool get_task(const FwdParams& p, bool causal, int idx, Task& t) {
  if (p.varlen) {
    if (idx >= *p.task_count) return false;
    const int4 e = p.tasks[idx];
    const int s0 = p.cu_seqlens[e.x], s1 = p.cu_seqlens[e.x + 1];
    const int k0 = p.cu_seqlens_k[e.x], k1 = p.cu_seqlens_k[e.x + 1];
    t.kvh = e.y & 0xffff; t.split = e.y >> 16; t.row0 = e.z * ROWS; t.rows = ROWS;
    t.tok0 = s0; t.len = s1 - s0;
    t.tok0k = k0; t.lenk = k1 - k0; t.off = t.lenk - t.len;
    t.lse_base = (t.kvh << p.gshift) * p.total_tokens + s0;
    t.lse_hstride = p.total_tokens;
    return true;
  }
  if (idx >= p.num_tasks) return false;
  t.split = idx % p.splits;   // the key ranges of one (b, kv head, m) are consecutive tasks
  idx /= p.splits;
  int bh, m;
  if (causal) {
    // Longest-processing-time order: heavy m-blocks first, inside sections of
    // lpt_group (b, kv head) pairs so that a section's K/V stays resident in L2
    // ("Flash Attention 4", section "Tile 调度"; "FlashAttention-4（下）", section "6. LPT 调度").
    const int bh_total = p.B * p.Hkv;
    const int per_group = p.lpt_group * p.num_m;
    const int g = idx / per_group;
    const int r = idx - g * per_group;
    const int gsize = min(p.lpt_group, bh_total - g * p.lpt_group);
    m = p.num_m - 1 - r / gsize;
    bh = g * p.lpt_group + r % gsize;
  } else {
    bh = idx / p.num_m;
    m = idx - bh * p.num_m;
  }
  const int b = bh / p.Hkv;
  t.kvh = bh - b * p.Hkv; t.row0 = m * ROWS; t.rows = ROWS; t.tok0 = b * p.N; t.len = p.N;
  t.tok0k = b * p.Nk; t.lenk = p.Nk; t.off = p.Nk - p.N + p.diag_shift;
  t.lse_base = (b * p.H + (t.kvh << p.gshift)) * p.N;
  t.lse_hstride = p.N;
  return true;
}

// Q tile 1 of the task holds no query row of the sequence (its packed rows
// start at or past the end), or the task is a solo one of 128 rows: the task runs
// Q tile 0 only. Decoding (a few query rows per sequence) and the ragged last block
// of a sequence are such tasks.
__device__ __forceinline__ bool task_one_tile(const Task& t, int gshift) {
  return t.rows == kBlockM || packed_pos(t, kBlockM, gshift) >= t.len;
}

// Causal offset: query position i sees keys j <= i + off, with off = N_kv - N_q
// (bottom-right alignment, "Flash Attention 4", section "Causal Mask"); a key shard
// adds the keys that follow it in the full sequence.
__device__ __forceinline__ int task_off(const Task& t) { return t.off; }

// K/V blocks [lo, hi) a task visits, from hi - 1 down to lo. Causal work stops
// at the last key the bottom row of the task may see; with splits > 1 the
// sequence's blocks are cut into `splits` ranges of ceil(blocks / splits) and
// the task keeps its range's share. hi <= lo: the task sees no key.
struct KRange {
  int lo, hi;
};
// The same for the packed rows [row0, row0 + rows) of a sequence with lenk key rows and
// causal offset off.
__device__ __forceinline__ KRange key_range(int row0, int rows, int off, int lenk, int gshift, bool causal,
                                            int splits, int split) {
  int kmax = lenk;
  if (causal) kmax = min(((row0 + rows - 1) >> gshift) + off + 1, lenk);
  const int nb = kmax > 0 ? (kmax + kBlockN - 1) / kBlockN : 0;
  if (splits == 1) return {0, nb};
  const int per = ((lenk + kBlockN - 1) / kBlockN + splits - 1) / splits;
  const int lo = split * per;
  return {lo, max(lo, min(lo + per, nb))};
}
__device__ __forceinline__ KRange task_range(const FwdParams& p, const Task& t, bool causal) {
  return key_range(t.row0, t.rows, t.off, t.lenk, p.gshift, causal, p.splits, t.split);
}

// ------------------------------------------------------------------ task ring
// The producer warp claims task indices and publishes them (or -1 = no more
// work) through a two-slot ring in shared memory. The MMA warp, the 8 softmax
// warps and the 4 correction warps take the k-th task from slot k % 2 and give
// the slot back with one arrival per warp.
constexpr int kTaskConsumerWarps = 13;

// Causal tasks: the top K/V block lies entirely above Q tile 0's last row, so
// tile 0 skips it (its scores there would all be masked). Returns 1 or 0.
// (A solo task's range already ends at its only tile's last visible key.)
__device__ __forceinline__ int task_skip0(const Task& t, KRange r, bool causal, int gshift) {
  return (causal && t.rows != kBlockM && r.hi - r.lo >= 2 &&
          (r.hi - 1) * kBlockN > packed_pos(t, kBlockM - 1, gshift) + task_off(t))
             ? 1 : 0;
}

// ------------------------------------------------------------------ bounded waits
struct Waiter {
  volatile int* abort_flag;
  unsigned long long timeout_ns;
  uint32_t role;

  // Called by all 32 lanes of a warp together; the result is warp-uniform (every
  // lane has observed the phase, so each has its own acquire).
  __device__ __forceinline__ bool wait(uint32_t bar_addr, uint32_t parity, uint32_t bar_id, int block) {
    uint64_t t0 = 0;
    for (uint32_t it = 0;; ++it) {
      if (__all_sync(0xffffffffu, mbar_try_wait(bar_addr, parity))) return true;
      if ((it & 63) == 63) {
        if (__any_sync(0xffffffffu, *abort_flag != 0)) return false;
        const uint64_t now = __shfl_sync(0xffffffffu, globaltimer(), 0);
        if (t0 == 0) t0 = now;
        else if (now - t0 > timeout_ns) {
          give_up(bar_id, block);
          return false;
        }
      }
    }
  }
  // For loops that poll several barriers in turn: call once per round; returns
  // false (after recording a timeout once the limit has passed) when the loop
  // must give up. Warp-uniform like wait().
  __device__ __forceinline__ bool still_waiting(uint32_t& it, uint64_t& t0, uint32_t bar_id, int block) {
    if ((++it & 63) != 0) return true;
    if (__any_sync(0xffffffffu, *abort_flag != 0)) return false;
    const uint64_t now = __shfl_sync(0xffffffffu, globaltimer(), 0);
    if (t0 == 0) {
      t0 = now;
    } else if (now - t0 > timeout_ns) {
      give_up(bar_id, block);
      return false;
    }
    return true;
  }
  // Cold path: raise the CTA's abort flag and record the first timeout.
  __device__ __noinline__ void give_up(uint32_t bar_id, int block) {
    *abort_flag = 1;
    const unsigned long long word = kStatusTimeout | ((unsigned long long)role << 8) |
                                    ((unsigned long long)bar_id << 16) |
                                    ((unsigned long long)(uint32_t)block << 32);
    atomicCAS(&g_fa_status, 0ull, word);
  }
};

// ------------------------------------------------------------------ packed fp32 pairs (f32x2)
__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void unpack2(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.ftz.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.ftz.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
template <bool F16>
__device__ __forceinline__ uint32_t pack_16x2_u64(uint64_t v) {
  float lo, hi;
  unpack2(v, lo, hi);
  return pack_16x2<F16>(lo, hi);
}
// Rounding error of one weight as the PV product sees it: round(p) - p, with round the
// conversion to the 16-bit type of P (round to nearest even). Exact in fp32.
template <bool F16>
__device__ __forceinline__ float p_rounding_error(float p) {
  const uint32_t h = pack_16x2<F16>(p, 0.f) & 0xffffu;
  float r;
  if constexpr (F16) {
    asm("{\n\t.reg .f16 t;\n\tmov.b16 t, %1;\n\tcvt.f32.f16 %0, t;\n\t}" : "=f"(r) : "h"((unsigned short)h));
  } else {
    r = __uint_as_float(h << 16);
  }
  return r - p;
}
// The same weight computed as the exponential loop computes the block maximum's:
// exp2(m * sl2 - ref * sl2) with one fused multiply-add and the hardware ex2.
__device__ __forceinline__ float p_of_score(float m, float sl2, float bias) {
  float x;
  asm("fma.rn.ftz.f32 %0, %1, %2, %3;" : "=f"(x) : "f"(m), "f"(sl2), "f"(bias));
  return ex2_approx(x);
}
__device__ __forceinline__ float max3(float a, float b, float c) {
  float m;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(m) : "f"(a), "f"(b), "f"(c));
  return m;
}
// ------------------------------------------------------------------ exp2 on the FMA pipe
// 2^x = 2^j * p(f) with j = round(x), f = x - j in [-1/2, 1/2] and p a cubic
// fitted to 2^f by the Remez exchange algorithm (all four coefficients free,
// max relative error 7.5e-5; see fit_exp2_poly.py). Rounding uses the 1.5*2^23
// trick: in x + 1.5*2^23 the low mantissa bits hold round(x), and shifting that
// word left by 23 moves j into the exponent field. No instruction of this path
// runs on the transcendental (XU) pipe. x is clamped to [-126, 126] so the
// exponent field stays in range: inputs below -126 give a non-negative value
// under 2^-125 instead of 0, inputs above 126 give 2^126 * p(f) instead of inf.
// ("Flash Attention 4", section "算法结构": part of the exponentials run as a
// cubic polynomial on FMA units so the hardware ex2 unit is not the only path.)
constexpr float kRoundMagic = 12582912.0f;  // 1.5 * 2^23
constexpr float kP0 = 0.9999280571937561f, kP1 = 0.6932609677314758f, kP2 = 0.2426111251115799f,
                kP3 = 0.0551716685295105f;

__device__ __forceinline__ float exp2_poly(float x) {
  x = fminf(fmaxf(x, -126.0f), 126.0f);
  const float r = __fadd_rn(x, kRoundMagic);
  const float f = __fsub_rn(x, __fsub_rn(r, kRoundMagic));
  float q = fmaf(f, kP3, kP2);
  q = fmaf(q, f, kP1);
  q = fmaf(q, f, kP0);
  return __int_as_float(__float_as_int(q) + (__float_as_int(r) << 23));
}

// The same steps on a pair, with the adds and the Horner steps as f32x2 ops.
__device__ __forceinline__ uint64_t exp2_poly2(uint64_t x2) {
  float x0, x1;
  unpack2(x2, x0, x1);
  const uint64_t x = pack2(fminf(fmaxf(x0, -126.0f), 126.0f), fminf(fmaxf(x1, -126.0f), 126.0f));
  const uint64_t r = add2(x, pack2(kRoundMagic, kRoundMagic));
  const uint64_t f = fma2(add2(r, pack2(-kRoundMagic, -kRoundMagic)), pack2(-1.0f, -1.0f), x);
  uint64_t q = fma2(f, pack2(kP3, kP3), pack2(kP2, kP2));
  q = fma2(q, f, pack2(kP1, kP1));
  q = fma2(q, f, pack2(kP0, kP0));
  float q0, q1, r0, r1;
  unpack2(q, q0, q1);
  unpack2(r, r0, r1);
  return pack2(__int_as_float(__float_as_int(q0) + (__float_as_int(r0) << 23)),
               __int_as_float(__float_as_int(q1) + (__float_as_int(r1) << 23)));
}

// The block maximum's weight as an emulated column computes it (the pair path, low lane).
__device__ __forceinline__ float p_of_score_poly(float m, float sl2, float bias) {
  float x;
  asm("fma.rn.ftz.f32 %0, %1, %2, %3;" : "=f"(x) : "f"(m), "f"(sl2), "f"(bias));
  float lo, hi;
  unpack2(exp2_poly2(pack2(x, x)), lo, hi);
  return lo;
}

// ------------------------------------------------------------------ MMA issue helpers
// S = Q K^T : M = 128 rows, N = 128 keys, K = D (16 per instruction). Both
// operands K-major with 128-byte swizzle; a K step of 16 elements is a 32-byte
// advance inside a 128-byte row; D = 128 spans two 64-column slabs.
// qdesc / kdesc: descriptors of the tiles' first byte; the per-step offsets are
// added to the 16-byte start-address field (shared-memory addresses stay below
// 256 KiB, so the 14-bit field never carries).
template <int D, bool F16>
__device__ __forceinline__ void issue_qk(uint32_t d_tmem, uint64_t qdesc, uint64_t kdesc) {
  constexpr uint32_t idesc = idesc_f32acc(128, kBlockN, false, F16);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint32_t off = ((kk / 4) * Layout<D>::kSlabBytes + (kk % 4) * 32) >> 4;
    mma_ss(d_tmem, qdesc + off, kdesc + off, idesc, kk > 0 ? 1u : 0u);
  }
}
// O (+)= P V : M = 128 rows, N = D, K = 128 keys. P (16-bit pairs) from TMEM,
// 8 columns per 16 keys. V is [keys, d] in smem = MN-major for the B operand:
// 64-wide d slabs LBO = 16 KiB apart, 8-key groups SBO = 1 KiB apart; a K step
// of 16 keys is a 2 KiB advance.
// vdesc: MN-major descriptor of the V tile's first byte (LBO = one 64-column slab).
template <int D, int K0, int K1, bool F16>
__device__ __forceinline__ void issue_pv(uint32_t d_tmem, uint32_t p_tmem, uint64_t vdesc, bool accumulate) {
  constexpr uint32_t idesc = idesc_f32acc(128, D, true, F16);
#pragma unroll
  for (int kk = K0 / 16; kk < K1 / 16; ++kk)
    mma_ts(d_tmem, p_tmem + kk * 8, vdesc + ((kk * 2048) >> 4), idesc, (accumulate || kk > 0) ? 1u : 0u);
}

// ------------------------------------------------------------------ the kernel
// SOLO: tasks of one 128-row Q tile whose score tile alternates between
// S_0 and S_1 (the host launches it when p.task_rows == 128).
template <int D, bool CAUSAL, bool EMU, bool F16, bool SOLO = false>
__global__ void __launch_bounds__(kThreads, 1) fa_fwd_kernel(const __grid_constant__ FwdParams p) {
  constexpr int kRows = SOLO ? kBlockM : kTaskRows;   // packed rows per task
  using L = Layout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sQ = sbase + L::kQOff;
  const uint32_t sKV = sbase + L::kKVOff;
  const uint32_t sOst = sbase + L::kOstOff;
  const uint32_t sBar = sbase + L::kBarOff;
  float* mail = reinterpret_cast<float*>(smem + L::kMailOff);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 4);
  volatile int* never_abort = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 8);  // stays 0
  volatile int* task_slot = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 16);   // [2]
  const uint32_t clc_resp = sbase + L::kClcOff;
  auto bar = [&](int i) -> uint32_t { return sBar + 8u * (uint32_t)i; };

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  // ---- setup
  if (tid == 0) {
    *abort_flag = 0;
    *never_abort = 0;
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(L::bQFull + i), 1);
      mbar_init(bar(L::bQEmpty + i), 1);
      mbar_init(bar(L::bSFull + i), 1);
      // two-tile tasks: first part of P stored (softmax) + O ready (WG2); solo tasks: both
      // warpgroups' halves of P stored + O ready
      mbar_init(bar(L::bPO + i), (SOLO ? 3 : 2) * kBlockM);
      mbar_init(bar(L::bP2 + i), kBlockM);          // two-tile tasks: the rest of P stored (softmax)
      mbar_init(bar(L::bCorrFull + i), kBlockM);
      mbar_init(bar(L::bCorrEmpty + i), kBlockM);
      mbar_init(bar(L::bOFinal + i), 1);
      mbar_init(bar(L::bTurn + i), kBlockM);        // the other softmax warpgroup's exponentials done
      mbar_init(bar(L::bStats + i), kBlockM);       // final row_sum in the mailbox (stats_tmem mode)
    }
    for (int s = 0; s < L::kStages; ++s) {
      mbar_init(bar(L::bKVFull + s), 1);
      mbar_init(bar(L::bKVEmpty + s), 1);
    }
    mbar_init(bar(L::bDrain), 1);
    mbar_init(bar(L::bPVDone), 1);   // solo tasks: one phase per key block, once its PV has completed
    for (int i = 0; i < 2; ++i) mbar_init(bar(L::bXchg + i), 2 * kBlockM);   // solo: partial maxima swapped
    mbar_init(bar(L::bRowSum), kBlockM);   // solo: WG1's row sums handed to WG0
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(L::bTaskFull + i), 1);
      mbar_init(bar(L::bTaskEmpty + i), kTaskConsumerWarps);
    }
    mbar_init(bar(L::bClc), 1);
    mbar_init(bar(L::bOstReady), kBlockM);
    mbar_init(bar(L::bOstFree), 1);
    fence_mbar_init();
  }
  if (warp == 13 && lane == 0) {
    prefetch_tmap(&p.tm_q);
    prefetch_tmap(&p.tm_k);
    prefetch_tmap(&p.tm_v);
    prefetch_tmap(&p.tm_o);
  }
  if (warp == 12) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // Launched with programmatic stream serialization, everything above may overlap
  // the previous kernel in the stream; global memory is touched only from here on.
  // (Only such launches execute the wait: in the others it measured 0.3-0.5 % slower.)
  if (p.pdl) griddep_wait();

  // consumers: the k-th task of this CTA from the ring (warp-uniform; -1 = done)
  auto take_task = [&](Waiter& w, int k) -> int {
    const int slot = k & 1;
    if (!w.wait(bar(L::bTaskFull + slot), (k >> 1) & 1, L::bTaskFull + slot, -1)) return -1;
    const int idx = task_slot[slot];
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(L::bTaskEmpty + slot));
    return idx;
  };

  // Register split 192/192/48/80 per thread for WG0/WG1/WG2/WG3 (sum = 4 x 128,
  // the launch allocation). Each setmaxnreg sits inside its role's branch so the
  // compiler allocates that role's code with the new limit.
  if (warp >= 12) setmaxnreg_dec<80>();
  if (warp == 13) {
    // ================================================================ TMA producer
    // The whole warp runs the loop (its state stays warp-uniform); one elected
    // lane issues the copies.
    {
      Waiter w{abort_flag, p.timeout_ns, kRoleLoad};
      Tracer tr;
      tr.init(p, 0, lane == 0);
      const bool leader = elect_one();
      uint32_t stage = 0, phase = 0;
      // armed full barriers and the parity of their last arm, for the drain on abort
      uint32_t q_armed = 0, q_par = 0, kv_armed = 0, kv_par = 0;
      uint32_t q_uses = 0;   // bit t: parity of the number of loads into Q slot t so far
      bool ok = true;
      auto load_tile = [&](const CUtensorMap* m, uint32_t dst, int tok, int h, uint32_t b) {
#pragma unroll
        for (int c = 0; c < L::kHalves; ++c) tma_load_3d(dst + c * L::kSlabBytes, m, c * 64, h, tok, b);
      };
      auto load_kv = [&](const CUtensorMap* m, int tok, int h, int blk) -> bool {
        if (!w.wait(bar(L::bKVEmpty + stage), phase ^ 1, L::bKVEmpty + stage, blk)) return false;
        if (leader) {
          mbar_arrive_expect_tx(bar(L::bKVFull + stage), L::kTileBytes);
          load_tile(m, sKV + stage * L::kTileBytes, tok, h, bar(L::bKVFull + stage));
        }
        __syncwarp();
        tr.rec(m == &p.tm_k ? kEvK : kEvV, blk);
        kv_armed |= 1u << stage;
        kv_par = (kv_par & ~(1u << stage)) | (phase << stage);
        if (++stage == L::kStages) { stage = 0; phase ^= 1; }
        return true;
      };
      auto load_q = [&](int t, int tok, int h, int blk) -> bool {
        const uint32_t use = (q_uses >> t) & 1u;
        if (!w.wait(bar(L::bQEmpty + t), use ^ 1u, L::bQEmpty + t, blk)) return false;
        if (leader) {
          mbar_arrive_expect_tx(bar(L::bQFull + t), L::kTileBytes);
          load_tile(&p.tm_q, sQ + t * L::kTileBytes, tok, h, bar(L::bQFull + t));
        }
        __syncwarp();
        tr.rec(t == 0 ? kEvQ0 : kEvQ1, blk);
        q_armed |= 1u << t;
        q_par = (q_par & ~(1u << t)) | (use << t);
        q_uses ^= 1u << t;
        return true;
      };
      // The producer also claims this CTA's tasks and publishes them to the other
      // warps: sched 2 takes over the task of a CTA that has not been launched
      // yet (cluster launch control), which turns the launch order (longest task
      // first for causal work) into a dynamic work queue; it does so only after
      // issuing the last load of the current task, so a task is claimed shortly
      // before an SM is free for it. sched 1 strides by the grid size; sched 0
      // runs only blockIdx.x.
      const int limit = p.varlen ? *p.task_count : p.num_tasks;
      uint32_t clc_par = 0;
      auto claim_next = [&](int cur) -> int {
        for (;;) {
          int n;
          if (p.sched == 2) {
            if (leader) {
              mbar_arrive_expect_tx(bar(L::bClc), 16);
              clc_try_cancel(clc_resp, bar(L::bClc));
            }
            __syncwarp();
            if (!w.wait(bar(L::bClc), clc_par, L::bClc, -1)) return -1;
            clc_par ^= 1;
            n = clc_cancelled_ctaid_x(clc_resp);
          } else {
            n = p.sched == 1 ? cur + (int)gridDim.x : -1;
          }
          if (n < limit) return n;       // includes n = -1: no more work
          if (p.sched != 2) return -1;   // static orders only grow
          cur = n;                       // a grid-padding CTA without work: keep claiming
        }
      };
      int idx = (int)blockIdx.x;
      Task tk;
      for (int k = 0; ok; ++k) {
        if (k > 0 || idx >= limit) idx = claim_next(idx);
        const int slot = k & 1;
        if (!w.wait(bar(L::bTaskEmpty + slot), ((k >> 1) & 1) ^ 1, L::bTaskEmpty + slot, -1)) { ok = false; break; }
        if (leader) {
          task_slot[slot] = idx;
          mbar_arrive(bar(L::bTaskFull + slot));
        }
        __syncwarp();
        if (idx < 0) {
          // no task left to claim (none of the grid's CTAs waits to launch): the next
          // kernel in the stream may start its prologue on the SMs this grid frees
          if (leader && p.pdl) griddep_launch_dependents();
          break;
        }
        get_task<kRows>(p, CAUSAL, idx, tk);
        const KRange kr = task_range(p, tk, CAUSAL);
        if (kr.hi <= kr.lo) continue;   // no key to attend to: nothing to load
        const int nb = kr.hi - kr.lo;
        const bool one = task_one_tile(tk, p.gshift);
        // load order: Q_0, K_{hi-1}, Q_1, V_{hi-1}, K_{hi-2}, V_{hi-2}, ..., K_lo, V_lo
        // (Q tile t: positions from packed_pos(t * 128) of query heads kvh*G .. kvh*G+G-1;
        // no Q_1 when tile 1 has no row)
#pragma unroll 1
        for (int e = 0; ok && e < 2 * nb + 2; ++e) {
          if (e == 0 || e == 2) {
            const int t = e >> 1;
            if (t == 1 && one) continue;
            ok = load_q(t, tk.tok0 + packed_pos(tk, t * kBlockM, p.gshift), tk.kvh << p.gshift, kr.hi - 1);
          } else {
            const int kvi = e == 1 ? 0 : e - 2;          // even: K, odd: V
            const int j = kr.hi - 1 - (kvi >> 1);
            ok = load_kv((kvi & 1) ? &p.tm_v : &p.tm_k, tk.tok0k + j * kBlockN, tk.kvh, j);
          }
        }
      }
      if (!ok) {
        // drain: every armed full barrier completes once its bytes have landed
        Waiter d{never_abort, p.timeout_ns, kRoleDrain};
#pragma unroll 1
        for (int t = 0; t < 2; ++t)
          if (q_armed & (1u << t)) d.wait(bar(L::bQFull + t), (q_par >> t) & 1, L::bQFull + t, -1);
#pragma unroll 1
        for (int s = 0; s < L::kStages; ++s)
          if (kv_armed & (1u << s)) d.wait(bar(L::bKVFull + s), (kv_par >> s) & 1, L::bKVFull + s, -1);
      }
    }
  } else if (warp == 12) {
    // ================================================================ MMA issuer
    // The whole warp runs the loop so stages, phases and descriptors stay in
    // uniform registers; one elected lane (the same one throughout, so its
    // tcgen05.commit covers its own MMAs) issues the tcgen05 instructions.
    {
      Waiter w{abort_flag, p.timeout_ns, kRoleMma};
      Tracer tr;
      tr.init(p, 1, lane == 0);
      const bool leader = elect_one();
      uint32_t stage = 0, phase = 0;
      uint32_t po_par = 0, p2_par = 0;  // bit t: parity of the next wait on p_o[t] / p2[t]
      uint32_t qf_par = 0;              // bit t: parity of the next wait on q_full[t]
      bool ok = true;
      const uint32_t S0 = tmem + L::col_s(0), S1 = tmem + L::col_s(1);
      const uint32_t O0 = tmem + L::col_o(0), O1 = tmem + L::col_o(1);
      const uint32_t P0 = S0 + 64, P1 = S1 + 64;
      const uint64_t Q0 = smem_desc_sw128(sQ, 16, 1024), Q1 = smem_desc_sw128(sQ + L::kTileBytes, 16, 1024);
      const uint64_t Kd = smem_desc_sw128(sKV, 16, 1024);              // K tile of stage 0 (K-major)
      const uint64_t Vd = smem_desc_sw128(sKV, L::kSlabBytes, 1024);   // V tile of stage 0 (MN-major)
      constexpr uint32_t kStageStep = L::kTileBytes >> 4;
      Task tk;
      for (int k = 0; ok; ++k) {
        const int idx = take_task(w, k);
        if (idx < 0) break;
        get_task<kRows>(p, CAUSAL, idx, tk);
        const KRange kr = task_range(p, tk, CAUSAL);
        if (kr.hi <= kr.lo) continue;   // no key: no MMA (the epilogue writes the empty rows)
        const int nb = kr.hi - kr.lo;
        if constexpr (SOLO) {
          // Solo task: one Q tile whose score tile alternates between S_0 (even blocks i)
          // and S_1 (odd), so block i+2's QK^T, issued as soon as PV_i has read P_i out of
          // the same columns, runs while the softmax works on block i+1. The task's K/V
          // items in ring order are K_{hi-1}, V_{hi-1}, K_{hi-2}, ...: item 2i is block
          // i's K, item 2i+1 its V; the K items are used two blocks ahead of the V items.
          // Step i issues PV_i (i >= 0) and then QK_{i+2}.
          const uint32_t c0 = phase * L::kStages + stage;   // ring position of the task's first item
#pragma unroll 1
          for (int i = -2; i < nb; ++i) {
            if (i >= 0) {
              const int b = i & 1, j = kr.hi - 1 - i;
              const uint32_t c = (c0 + 2u * (uint32_t)i + 1u) % (2u * L::kStages);
              const uint32_t vs = c % L::kStages;
              if (!w.wait(bar(L::bKVFull + vs), c / L::kStages, L::bKVFull + vs, j)) { ok = false; break; }
              // both halves of P (the warpgroups finish within ~150 cycles of each other)
              // and O: one wait
              if (!w.wait(bar(L::bPO + b), (po_par >> b) & 1, L::bPO + b, j)) { ok = false; break; }
              po_par ^= 1u << b;
              tc_fence_after();
              // P of keys 0-63 in columns [0, 32) of the score tile, of keys 64-127 in [64, 96)
              if (leader) {
                issue_pv<D, 0, kSoloSplitP, F16>(O0, b ? S1 : S0, Vd + vs * kStageStep, i > 0);
                issue_pv<D, kSoloSplitP, kBlockN, F16>(O0, (b ? S1 : S0) + 32, Vd + vs * kStageStep, true);
                mma_commit(bar(L::bKVEmpty + vs));
                mma_commit(bar(L::bPVDone));                         // O holds blocks 0 .. i
                if (i == nb - 1) mma_commit(bar(L::bOFinal + 0));
              }
              __syncwarp();
              tr.rec(kEvPV0b, j);
            }
            const int n = i + 2;   // S_(n&1) = Q K_n^T
            if (n < nb) {
              const uint32_t c = (c0 + 2u * (uint32_t)n) % (2u * L::kStages);
              const uint32_t ks_ = c % L::kStages;
              if (!w.wait(bar(L::bKVFull + ks_), c / L::kStages, L::bKVFull + ks_, kr.hi - 1 - n)) { ok = false; break; }
              if (n == 0) {
                if (!w.wait(bar(L::bQFull + 0), qf_par & 1u, L::bQFull + 0, kr.hi - 1)) { ok = false; break; }
                qf_par ^= 1u;
              }
              tc_fence_after();
              if (leader) {
                issue_qk<D, F16>((n & 1) ? S1 : S0, Q0, Kd + ks_ * kStageStep);
                mma_commit(bar(L::bSFull + (n & 1)));
                mma_commit(bar(L::bKVEmpty + ks_));
                if (n == nb - 1) mma_commit(bar(L::bQEmpty + 0));   // Q_0's last use in this task
              }
              __syncwarp();
              tr.rec(kEvS0 + (n & 1), kr.hi - 1 - n);
            }
          }
          if (!ok) break;
          const uint32_t c = (c0 + 2u * (uint32_t)nb) % (2u * L::kStages);   // past the task's items
          stage = c % L::kStages;
          phase = c / L::kStages;
          continue;
        }
        const int skip0 = task_skip0(tk, kr, CAUSAL, p.gshift);   // tile 0 starts one block lower
        const int t_last = task_one_tile(tk, p.gshift) ? 0 : 1;   // the tiles of this task: 0 .. t_last
        // prologue: S_0 and S_1 for the top block (S_0 only if tile 0 sees it)
        uint32_t ks = stage;
        if (!w.wait(bar(L::bKVFull + ks), phase, L::bKVFull + ks, kr.hi - 1)) { ok = false; break; }
        if (++stage == L::kStages) { stage = 0; phase ^= 1; }
#pragma unroll 1
        for (int t = 0; t <= t_last; ++t) {
          if (!w.wait(bar(L::bQFull + t), (qf_par >> t) & 1, L::bQFull + t, nb - 1)) { ok = false; break; }
          qf_par ^= 1u << t;
          tc_fence_after();
          tr.rec(kEvIssueBegin, 0);
          if (leader) {
            if (t == 1 || !skip0) {
              issue_qk<D, F16>(t ? S1 : S0, t ? Q1 : Q0, Kd + ks * kStageStep);
              mma_commit(bar(L::bSFull + t));
            }
            if (t == t_last) mma_commit(bar(L::bKVEmpty + ks));
            if (nb == 1) mma_commit(bar(L::bQEmpty + t));   // Q_t's last use: the next task's Q may load
          }
          __syncwarp();
          tr.rec(kEvS0 + t, kr.hi - 1);
        }
        if (!ok) break;
        for (int i = 0; i < nb; ++i) {
          const int j = kr.hi - 1 - i;
          const bool last = (i == nb - 1);
          const uint32_t vs = stage;
          if (!w.wait(bar(L::bKVFull + vs), phase, L::bKVFull + vs, j)) { ok = false; break; }
          tr.rec(kEvKVV, j);
          if (++stage == L::kStages) { stage = 0; phase ^= 1; }
          // per Q tile t: O_t (+)= P_t V_j in two halves, then S_t for block j-1
#pragma unroll 1
          for (int t = 0; t <= t_last; ++t) {
            const uint32_t Ot = t ? O1 : O0, Pt = t ? P1 : P0, St = t ? S1 : S0;
            const uint64_t Qt = t ? Q1 : Q0;
            const int first_i = t == 0 ? skip0 : 0;   // this tile's first block
            if (i >= first_i) {
              if (!w.wait(bar(L::bPO + t), (po_par >> t) & 1, L::bPO + t, j)) { ok = false; break; }
              po_par ^= 1u << t;
              tr.rec(kEvPO0 + 4 * t, j);
              tc_fence_after();
              tr.rec(kEvIssueBegin, 0);
              if (leader) issue_pv<D, 0, kSplitP, F16>(Ot, Pt, Vd + vs * kStageStep, i > first_i);
              tr.rec(kEvPV0a + 4 * t, j);
              if (!w.wait(bar(L::bP2 + t), (p2_par >> t) & 1, L::bP2 + t, j)) { ok = false; break; }
              p2_par ^= 1u << t;
              tr.rec(kEvP20 + 4 * t, j);
              tc_fence_after();
              tr.rec(kEvIssueBegin, 0);
              if (leader) issue_pv<D, kSplitP, kBlockN, F16>(Ot, Pt, Vd + vs * kStageStep, true);
              tr.rec(kEvPV0b + 4 * t, j);
            }
            if (t == t_last && leader) mma_commit(bar(L::bKVEmpty + vs));   // V_j read by the task's tiles
            if (!last) {
              if (t == 0) {
                ks = stage;
                if (!w.wait(bar(L::bKVFull + ks), phase, L::bKVFull + ks, j - 1)) { ok = false; break; }
                tr.rec(kEvKVK, j - 1);
                if (++stage == L::kStages) { stage = 0; phase ^= 1; }
                tc_fence_after();
              }
              tr.rec(kEvIssueBegin, 0);
              if (leader) {
                issue_qk<D, F16>(St, Qt, Kd + ks * kStageStep);
                mma_commit(bar(L::bSFull + t));
                if (t == t_last) mma_commit(bar(L::bKVEmpty + ks));      // K_{j-1} read by the task's tiles
                if (j - 1 == kr.lo) mma_commit(bar(L::bQEmpty + t));     // last use of Q_t in this task
              }
              tr.rec(kEvS0 + t, j - 1);
            } else if (leader) {
              mma_commit(bar(L::bOFinal + t));
            }
            __syncwarp();
          }
          if (!ok) break;
        }
      }
      // all issued MMAs must finish before the tensor memory is released
      if (leader) mma_commit(bar(L::bDrain));
      Waiter d{never_abort, p.timeout_ns, kRoleDrain};
      d.wait(bar(L::bDrain), 0, L::bDrain, -1);
    }
  } else if (warp < 8) {
    // ================================================================ softmax WG0 / WG1
    setmaxnreg_inc<192>();
    const int t = warp >> 2;                 // Q tile of this warpgroup
    const int r = tid & 127;                 // row within the tile == TMEM lane
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_base + L::col_s(t);   // two-tile tasks: this warpgroup's score tile
    const uint32_t tP = tS + 64;
    Waiter w{abort_flag, p.timeout_ns, t == 0 ? kRoleSoftmax0 : kRoleSoftmax1};
    Tracer tr;
    tr.init(p, 2 + t, r == 0);
    const float sl2 = p.scale_log2;
    uint32_t s_par = 0, ce_par = 0;   // parity of the next wait on s_full / corr_empty (solo: bit b for [b])
    uint32_t turns = 0;   // exponential phases taken in turn so far (stagger mode)
    uint32_t x_par = 0, rs_par = 0;   // solo: bit b: next wait on xchg[b]; bit 0: on row_sum
    // Stagger mode ("Flash Attention 4", section "论文与当前 TIRx 实现的差异": the two
    // softmax warpgroups' exponential phases do not overlap): the warpgroups pass a
    // turn back and forth through bTurn, WG0 first. In a task of both tiles each takes
    // nb turns (WG0's first turn is an empty pass when tile 0 skips the top block),
    // so the turn is back at WG0 when the task ends.
    auto take_turn = [&](int j) -> bool {
      const uint32_t par = t == 0 ? (turns & 1u) ^ 1u : turns & 1u;
      ++turns;
      return w.wait(bar(L::bTurn + t), par, L::bTurn + t, j);
    };
    bool ok = true;
    Task tk;
    for (int k = 0; ok; ++k) {
      const int idx = take_task(w, k);
      if (idx < 0) break;
      get_task<kRows>(p, CAUSAL, idx, tk);
      const KRange kr = task_range(p, tk, CAUSAL);
      const int tile_pos0 = packed_pos(tk, t * kBlockM, p.gshift);  // sequence position of row 0
      const int pos = tile_pos0 + (r >> p.gshift);                  // this row's sequence position
      const int off = task_off(tk);
      // LSE of this row (split mode: of its key range) -> global memory
      auto store_lse = [&](float v) {
        if (pos < tk.len && tk.tok0 + pos < p.total_tokens) {
          const int li = tk.lse_base + (r & ((1 << p.gshift) - 1)) * tk.lse_hstride + pos;
          if (p.part_out) p.lse_part[tk.split * p.lse_split_stride + li] = v;
          else if (p.lse != nullptr) p.lse[li] = v;
        }
      };
      if constexpr (SOLO) {
        // Solo task: both warpgroups work on the one Q tile, warpgroup t on key columns
        // [64 t, 64 t + 64) of every block (half a softmax each). Per block they swap
        // their partial row maxima through shared memory (slot b = i & 1 of the second
        // Q buffer, unused by solo tasks) and take the same reference and acc_scale; each
        // keeps the row sum of its own columns, and WG1 hands its sum to WG0 at the end.
        // P of WG0's keys goes to columns [0, 32) of the score tile and WG1's to
        // [64, 96) (columns each has itself read); WG0 passes acc_scale in column 32.
        // Both warpgroups announce their half on p_o[b], which WG2's O arrival completes.
        float* xm = reinterpret_cast<float*>(smem + L::kQOff + L::kTileBytes);   // [2 blocks][2 halves][128]
        float* ysum = xm + 4 * kBlockM;                                          // [128] WG1's row sums
        if (kr.hi <= kr.lo) {   // no key for any row of the task: LSE = -inf (O = 0 is written by WG2)
          if (t == 0) store_lse(-INFINITY);
          continue;
        }
        const int nb = kr.hi - kr.lo;
        const int c0 = t * 64;   // this warpgroup's first key column of a block
        const int tp0 = packed_pos(tk, 0, p.gshift);   // both warpgroups: the rows of Q tile 0
        const int row_limit = CAUSAL ? min(tp0 + (r >> p.gshift) + off + 1, tk.lenk) : tk.lenk;  // keys [0, row_limit)
        float row_max = -INFINITY, row_sum = 0.f;
        float row_corr = 0.f;   // rounding errors of the blocks' largest weights (as in two-tile tasks)
        for (int i = 0; i < nb; ++i) {
          const int j = kr.hi - 1 - i, b = i & 1;
          const uint32_t tS = tmem + lane_base + L::col_s(b);
          if (!w.wait(bar(L::bSFull + b), (s_par >> b) & 1, L::bSFull + b, j)) { ok = false; break; }
          s_par ^= 1u << b;
          tr.rec(kEvSFull, j);
          tc_fence_after();
          const int k0 = j * kBlockN + c0;   // key of this warpgroup's first column
          const bool need_mask = (k0 + 64 > tk.lenk) || (CAUSAL && k0 + 63 > tp0 + off);
          const int lim = need_mask ? row_limit - k0 : 64;   // columns [lim, 64) are masked
          float s[64];
          uint32_t u[64];
          tmem_ld32(tS + c0, *reinterpret_cast<uint32_t(*)[32]>(&u[0]));
          tmem_ld32(tS + c0 + 32, *reinterpret_cast<uint32_t(*)[32]>(&u[32]));
          tmem_wait_ld();
          float mx0 = -INFINITY, mx1 = -INFINITY;
          if (need_mask) {
#pragma unroll
            for (int c = 0; c < 64; c += 4) {
#pragma unroll
              for (int e = 0; e < 4; ++e) s[c + e] = (c + e < lim) ? __uint_as_float(u[c + e]) : -INFINITY;
              mx0 = max3(mx0, s[c], s[c + 1]);
              mx1 = max3(mx1, s[c + 2], s[c + 3]);
            }
          } else {
#pragma unroll
            for (int c = 0; c < 64; c += 4) {
#pragma unroll
              for (int e = 0; e < 4; ++e) s[c + e] = __uint_as_float(u[c + e]);
              mx0 = max3(mx0, s[c], s[c + 1]);
              mx1 = max3(mx1, s[c + 2], s[c + 3]);
            }
          }
          const float part = fmaxf(mx0, mx1);
          xm[(b * 2 + t) * kBlockM + r] = part;
          mbar_arrive(bar(L::bXchg + b));
          if (!w.wait(bar(L::bXchg + b), (x_par >> b) & 1, L::bXchg + b, j)) { ok = false; break; }
          x_par ^= 1u << b;
          const float blk_max = fmaxf(part, xm[(b * 2 + (t ^ 1)) * kBlockM + r]);
          tr.rec(kEvSMax, j);
          // delayed-rescale rule, on the whole row's maximum (the same in both warpgroups)
          float ref, acc;
          if (i == 0) {
            ref = blk_max;
            acc = 1.f;
          } else {
            const float cand = fmaxf(row_max, blk_max);
            const float cand_safe = cand == -INFINITY ? 0.f : cand;
            const float delta = (row_max - cand_safe) * sl2;
            if (delta >= -p.tau && row_max != -INFINITY) {
              ref = row_max;
              acc = 1.f;
            } else {
              ref = cand;
              acc = ex2_approx(delta);
            }
          }
          row_max = ref;
          if (i > 0 && t == 0) {   // acc_scale to WG2 before the exponentials
            if (p.stats_tmem) {
              tmem_st1(tS + 32, __float_as_uint(acc));
              tmem_wait_st();
              tc_fence_before();
            } else {
              if (!w.wait(bar(L::bCorrEmpty + b), ((ce_par >> b) & 1) ^ 1, L::bCorrEmpty + b, j)) { ok = false; break; }
              ce_par ^= 1u << b;
              mail[b * kBlockM + r] = acc;
            }
            mbar_arrive(bar(L::bCorrFull + b));
            tr.rec(kEvMail, j);
          }
          const float ref_safe = ref == -INFINITY ? 0.f : ref;
          // the block maximum's weight, whichever half holds it (both warpgroups compute it;
          // WG0 hands the normaliser to WG2)
          row_corr = row_corr * acc + p_rounding_error<F16>(p_of_score(blk_max, sl2, -ref_safe * sl2));
          const uint64_t scale2 = pack2(sl2, sl2);
          const uint64_t bias2 = pack2(-ref_safe * sl2, -ref_safe * sl2);
          uint64_t sum2a = 0, sum2b = 0;
          uint32_t pk[32];
#pragma unroll
          for (int c = 0; c < 64; c += 2) {
            float x0, x1;
            unpack2(fma2(pack2(s[c], s[c + 1]), scale2, bias2), x0, x1);
            const uint64_t pp = pack2(ex2_approx(x0), ex2_approx(x1));
            if (c & 2) sum2b = add2(sum2b, pp); else sum2a = add2(sum2a, pp);
            pk[c >> 1] = pack_16x2_u64<F16>(pp);
          }
          tmem_st32(tS + (t == 0 ? 0 : 64), pk);
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(bar(L::bPO + b));
          tr.rec(t == 0 ? kEvHalf1 : kEvHalf2, j);
          float sa, sb;
          unpack2(add2(sum2a, sum2b), sa, sb);
          row_sum = row_sum * acc + (sa + sb);
        }
        if (!ok) break;
        if (t == 1) {   // this half's row sums to WG0
          ysum[r] = row_sum;
          mbar_arrive(bar(L::bRowSum));
          continue;
        }
        if (!w.wait(bar(L::bRowSum), rs_par & 1, L::bRowSum, -1)) { ok = false; break; }
        rs_par ^= 1u;
        row_sum += ysum[r];
        // final statistics to WG2 (the normaliser of O), LSE straight to global memory
        if (!w.wait(bar(L::bCorrEmpty + 0), (ce_par & 1) ^ 1, L::bCorrEmpty + 0, -1)) { ok = false; break; }
        ce_par ^= 1u;
        mail[r] = row_sum + row_corr;
        mbar_arrive(bar(p.stats_tmem ? L::bStats + 0 : L::bCorrFull + 0));
        tr.rec(kEvStats, -1);
        const float ref_safe = row_max == -INFINITY ? 0.f : row_max;
        store_lse(row_sum > 0.f ? (lg2_approx(row_sum) + ref_safe * sl2) * 0.69314718055994531f : -INFINITY);
        continue;
      }
      // two-tile task: this warpgroup runs Q tile t alone
      if (kr.hi <= kr.lo) {   // no key for any row of the task: LSE = -inf (O = 0 is written by WG2)
        store_lse(-INFINITY);
        continue;
      }
      if (t == 1 && task_one_tile(tk, p.gshift)) continue;   // this tile has no row of the sequence
      const int hi = kr.hi - (t == 0 ? task_skip0(tk, kr, CAUSAL, p.gshift) : 0);   // this tile's top block + 1
      const int nb = hi - kr.lo;
      const bool stagger = p.stagger != 0 && !task_one_tile(tk, p.gshift);
      if (stagger && hi < kr.hi) {   // tile 0 skips the top block: hand the first turn to WG1
        if (!take_turn(kr.hi - 1)) { ok = false; break; }
        mbar_arrive(bar(L::bTurn + 1));
      }
      const int row_limit = CAUSAL ? min(pos + off + 1, tk.lenk) : tk.lenk;  // keys [0, row_limit) visible
      float row_max = -INFINITY, row_sum = 0.f;
      // O is normalised by row_sum + row_corr: row_corr adds, per key block, the 16-bit
      // rounding error of the block's largest weight, so a row dominated by one key
      // divides that key's rounded weight (the one PV multiplies) by itself. Without it a
      // dominant weight 2^delta kept under the delayed-rescale rule (delta up to tau, not
      // an integer) leaves its bf16 rounding, up to 2^-8 relative, in O: up to |v| * 2^-8.
      // The LSE uses the fp32 row_sum, the exact denominator.
      float row_corr = 0.f;
#ifdef FA_TRACE
      uint32_t n_upd = 0, n_resc = 0;   // this row's later-block updates and O rescales
#endif
      for (int i = 0; i < nb; ++i) {
        const int j = hi - 1 - i;
        if (!w.wait(bar(L::bSFull + t), s_par & 1, L::bSFull + t, j)) { ok = false; break; }
        s_par ^= 1u;
        tr.rec(kEvSFull, j);
        tc_fence_after();
        const int k0 = j * kBlockN;
        const bool need_mask = (k0 + kBlockN > tk.lenk) || (CAUSAL && k0 + kBlockN - 1 > tile_pos0 + off);
        const int lim = need_mask ? row_limit - k0 : kBlockN;   // columns [lim, 128) are masked
        // S in two halves: the second half's TMEM load overlaps the first half's max
        float s[kBlockN];
        uint32_t u[kBlockN];
        tmem_ld32(tS, *reinterpret_cast<uint32_t(*)[32]>(&u[0]));
        tmem_ld32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&u[32]));
        tmem_wait_ld();
        tmem_ld32(tS + 64, *reinterpret_cast<uint32_t(*)[32]>(&u[64]));
        tmem_ld32(tS + 96, *reinterpret_cast<uint32_t(*)[32]>(&u[96]));
        float mx0 = -INFINITY, mx1 = -INFINITY;
        if (need_mask) {
          // diagonal / tail block: columns >= lim become -inf before the max
#pragma unroll
          for (int c = 0; c < 64; c += 4) {
#pragma unroll
            for (int e = 0; e < 4; ++e) s[c + e] = (c + e < lim) ? __uint_as_float(u[c + e]) : -INFINITY;
            mx0 = max3(mx0, s[c], s[c + 1]);
            mx1 = max3(mx1, s[c + 2], s[c + 3]);
          }
          tmem_wait_ld();
#pragma unroll
          for (int c = 64; c < kBlockN; c += 4) {
#pragma unroll
            for (int e = 0; e < 4; ++e) s[c + e] = (c + e < lim) ? __uint_as_float(u[c + e]) : -INFINITY;
            mx0 = max3(mx0, s[c], s[c + 1]);
            mx1 = max3(mx1, s[c + 2], s[c + 3]);
          }
        } else {
#pragma unroll
          for (int c = 0; c < 64; c += 4) {
#pragma unroll
            for (int e = 0; e < 4; ++e) s[c + e] = __uint_as_float(u[c + e]);
            mx0 = max3(mx0, s[c], s[c + 1]);
            mx1 = max3(mx1, s[c + 2], s[c + 3]);
          }
          tmem_wait_ld();
#pragma unroll
          for (int c = 64; c < kBlockN; c += 4) {
#pragma unroll
            for (int e = 0; e < 4; ++e) s[c + e] = __uint_as_float(u[c + e]);
            mx0 = max3(mx0, s[c], s[c + 1]);
            mx1 = max3(mx1, s[c + 2], s[c + 3]);
          }
        }
        const float blk_max = fmaxf(mx0, mx1);
        tr.rec(kEvSMax, j);
        // delayed-rescale rule
        float ref, acc;
        if (i == 0) {
          ref = blk_max;
          acc = 1.f;
        } else {
          const float cand = fmaxf(row_max, blk_max);
          const float cand_safe = cand == -INFINITY ? 0.f : cand;
          const float delta = (row_max - cand_safe) * sl2;
          // a row with no valid score yet (reference -inf) always adopts the candidate
          if (delta >= -p.tau && row_max != -INFINITY) {
            ref = row_max;
            acc = 1.f;
          } else {
            ref = cand;
            acc = ex2_approx(delta);
          }
#ifdef FA_TRACE
          ++n_upd;
          n_resc += (row_max != -INFINITY && acc < 1.f) ? 1u : 0u;
#endif
        }
        row_max = ref;
        // hand acc_scale to WG2 now, so the O rescale runs while P is computed
        if (i > 0) {
          if (p.stats_tmem) {
            // through column 0 of S_t (all of S is in registers): the next write to S_t
            // is the QK^T of block j-1, issued only after the PV that waits for WG2's
            // rescale, so the slot needs no empty barrier
            tmem_st1(tS, __float_as_uint(acc));
            tmem_wait_st();
            tc_fence_before();
          } else {
            if (!w.wait(bar(L::bCorrEmpty + t), (ce_par & 1) ^ 1, L::bCorrEmpty + t, j)) { ok = false; break; }
            ce_par ^= 1u;
            mail[t * kBlockM + r] = acc;
          }
          mbar_arrive(bar(L::bCorrFull + t));
          tr.rec(kEvMail, j);
        }
        if (stagger && !take_turn(j)) { ok = false; break; }
        const float ref_safe = ref == -INFINITY ? 0.f : ref;
        // P = exp2(S * sl2 - ref * sl2) -> 16-bit pairs; with EMU the first emu_groups
        // 16-column groups use the FMA polynomial (blocks without masked columns only)
        const int emu = (EMU && !need_mask) ? p.emu_groups : 0;
        {
          float pm = p_of_score(blk_max, sl2, -ref_safe * sl2);
          if constexpr (EMU) {
            // the block maximum's weight as its own column computes it: by the polynomial
            // if the maximum lies in an emulated group
            if (emu > 0) {
              float mxe = -INFINITY;
#pragma unroll
              for (int c = 0; c < kBlockN; ++c)
                if (c < emu * 16) mxe = fmaxf(mxe, s[c]);
              if (mxe == blk_max) pm = p_of_score_poly(blk_max, sl2, -ref_safe * sl2);
            }
          }
          row_corr = row_corr * acc + p_rounding_error<F16>(pm);
        }
        const uint64_t scale2 = pack2(sl2, sl2);
        const uint64_t bias2 = pack2(-ref_safe * sl2, -ref_safe * sl2);
        uint64_t sum2a = 0, sum2b = 0;
        uint32_t pk[kBlockN / 2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
          for (int g = (h ? kSplitP / 16 : 0); g < (h ? kBlockN / 16 : kSplitP / 16); ++g) {
            if (EMU && g < emu) {
#pragma unroll
              for (int e = 0; e < 16; e += 2) {
                const int c = g * 16 + e;
                const uint64_t pp = exp2_poly2(fma2(pack2(s[c], s[c + 1]), scale2, bias2));
                if (e & 2) sum2b = add2(sum2b, pp); else sum2a = add2(sum2a, pp);
                pk[c >> 1] = pack_16x2_u64<F16>(pp);
              }
            } else {
#pragma unroll
              for (int e = 0; e < 16; e += 2) {
                const int c = g * 16 + e;
                float x0, x1;
                unpack2(fma2(pack2(s[c], s[c + 1]), scale2, bias2), x0, x1);
                const uint64_t pp = pack2(ex2_approx(x0), ex2_approx(x1));
                if (e & 2) sum2b = add2(sum2b, pp); else sum2a = add2(sum2a, pp);
                pk[c >> 1] = pack_16x2_u64<F16>(pp);
              }
            }
          }
          // this part of P (keys [0, 96), then [96, 128)) over the upper half of S_t (all of S was read above)
          static_assert(kSplitP == 96, "P is stored as 48 + 16 columns");
          if (h == 0) {
            tmem_st32(tP, *reinterpret_cast<const uint32_t(*)[32]>(&pk[0]));
            tmem_st16(tP + 32, *reinterpret_cast<const uint32_t(*)[16]>(&pk[32]));
          } else {
            tmem_st16(tP + 48, *reinterpret_cast<const uint32_t(*)[16]>(&pk[48]));
          }
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(bar(h == 0 ? L::bPO + t : L::bP2 + t));
          tr.rec(h == 0 ? kEvHalf1 : kEvHalf2, j);
        }
        if (stagger) mbar_arrive(bar(L::bTurn + (t ^ 1)));   // the other warpgroup's turn
        float sa, sb;
        unpack2(add2(sum2a, sum2b), sa, sb);
        row_sum = row_sum * acc + (sa + sb);
      }
      if (!ok) break;
      // final statistics to WG2 (the normaliser of O), LSE straight to global memory
      if (!w.wait(bar(L::bCorrEmpty + t), (ce_par & 1) ^ 1, L::bCorrEmpty + t, -1)) { ok = false; break; }
      ce_par ^= 1u;
      mail[t * kBlockM + r] = row_sum + row_corr;
      // with acc_scale in tensor memory the per-block hand-offs have no empty barrier,
      // so the final one takes a barrier of its own: on corr_full it could complete a
      // second phase before WG2 has waited for the last block's
      mbar_arrive(bar(p.stats_tmem ? L::bStats + t : L::bCorrFull + t));
      tr.rec(kEvStats, -1);
      {
        const float ref_safe = row_max == -INFINITY ? 0.f : row_max;
        store_lse(row_sum > 0.f ? (lg2_approx(row_sum) + ref_safe * sl2) * 0.69314718055994531f : -INFINITY);
      }
#ifdef FA_TRACE
      // every CTA: row updates and rescales summed into the two words after the stamps
      if (p.trace != nullptr) {
        const uint32_t u = __reduce_add_sync(0xffffffffu, n_upd), rs = __reduce_add_sync(0xffffffffu, n_resc);
        if (lane == 0 && u != 0) {
          unsigned long long* tot = p.trace + (size_t)p.trace_ctas * kTraceRoles * kTraceSlots;
          atomicAdd(tot, (unsigned long long)u);
          atomicAdd(tot + 1, (unsigned long long)rs);
        }
      }
#endif
    }
  } else if (warp < 12) {
    // ================================================================ correction + epilogue (WG2)
    setmaxnreg_dec<48>();
    const int r = tid & 127;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    Waiter w{abort_flag, p.timeout_ns, kRoleCorr};
    Tracer tr;
    tr.init(p, 4, r == 0);
    uint32_t cf_par = 0, of_par = 0;  // bit t: parity of the next wait on corr_full[t] / o_final[t]
    uint32_t fs_par = 0;              // bit t: parity of the next wait on stats[t] (stats_tmem mode)
    uint32_t ost_n = 0;               // uses of the O staging tile so far
    uint32_t pv_done = 0;             // solo tasks: key blocks whose PV completion bPVDone has counted
    bool ok = true;
    Task tk;
    // O_0 and O_1 are free for the first task's first PV; later tasks get this
    // arrival right after the epilogue of the same tile (below), so the next
    // task's PV can start while the other tile is still being written out. Solo
    // tasks use O_0 only, their first PV always through p_o[0].
    mbar_arrive(bar(L::bPO + 0));
    if (!SOLO) mbar_arrive(bar(L::bPO + 1));
    for (int k = 0; ok; ++k) {
      const int idx = take_task(w, k);
      if (idx < 0) break;
      get_task<kRows>(p, CAUSAL, idx, tk);
      const KRange kr = task_range(p, tk, CAUSAL);
      if (kr.hi <= kr.lo) {
        // no key for any row of the task: O = 0 (its LSE = -inf comes from the softmax warps)
#pragma unroll 1
        for (int t = 0; t < tk.rows / kBlockM; ++t) {
          const int pos = packed_pos(tk, t * kBlockM, p.gshift) + (r >> p.gshift);
          const int head = (tk.kvh << p.gshift) + (r & ((1 << p.gshift) - 1));
          if (pos < tk.len && tk.tok0 + pos < p.total_tokens) {
            const size_t row = (size_t)(tk.tok0 + pos) * p.H + head;
            uint4* dst = p.part_out
                             ? reinterpret_cast<uint4*>(p.o_part + ((size_t)tk.split * p.total_tokens * p.H + row) * D)
                             : reinterpret_cast<uint4*>(p.o + row * D);
            const int n16 = p.part_out ? D / 4 : D / 8;   // 16-byte units per row
#pragma unroll 1
            for (int c = 0; c < n16; ++c) dst[c] = make_uint4(0u, 0u, 0u, 0u);
          }
        }
        continue;
      }
      const int nb = kr.hi - kr.lo;
      const int skip0 = task_skip0(tk, kr, CAUSAL, p.gshift);
      const int t_last = task_one_tile(tk, p.gshift) ? 0 : 1;   // the tiles of this task: 0 .. t_last
      constexpr bool solo = SOLO;   // one Q tile; block i's statistics come with score tile i & 1
      tr.rec(kEvTask, nb);
      for (int i = 1; ok && i < nb; ++i) {
        const int j = kr.hi - 1 - i;
#pragma unroll 1
        for (int t = 0; t <= t_last; ++t) {
          if (t == 0 && i - skip0 < 1) continue;   // tile 0's first block needs no correction
          const int b = solo ? (i & 1) : t;
          if (!w.wait(bar(L::bCorrFull + b), (cf_par >> b) & 1, L::bCorrFull + b, j)) { ok = false; break; }
          cf_par ^= 1u << b;
          tr.rec(kEvCorrFull + t, j);
          float a;
          if (p.stats_tmem) {
            tc_fence_after();
            // acc_scale: column 0 of the tile's score tile; solo tasks: column 32 (WG0's half)
            a = __uint_as_float(tmem_ld1(tmem + lane_base + L::col_s(b) + (solo ? 32u : 0u)));
            tmem_wait_ld();
          } else {
            a = mail[b * kBlockM + r];
            mbar_arrive(bar(L::bCorrEmpty + b));
          }
          if (__any_sync(0xffffffffu, a < 1.f)) {
            // a solo task's score tile for this block was ready before the previous
            // block's PV had finished: wait for that PV before touching O
            if (solo && !w.wait(bar(L::bPVDone), (pv_done + (uint32_t)i - 1u) & 1u, L::bPVDone, j)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t tO = tmem + lane_base + L::col_o(t);
#pragma unroll 1
            for (int c = 0; c < D / 16; ++c) {
              uint32_t u[16];
              tmem_ld16(tO + c * 16, u);
              tmem_wait_ld();
#pragma unroll
              for (int e = 0; e < 16; ++e) u[e] = __float_as_uint(__uint_as_float(u[e]) * a);
              tmem_st16(tO + c * 16, u);
            }
            tmem_wait_st();
          }
          tc_fence_before();
          mbar_arrive(bar(L::bPO + b));
          tr.rec(kEvCorrDone + t, j);
        }
      }
      if (!ok) break;
      if (solo) pv_done += (uint32_t)nb;
      // epilogue: O_t / row_sum -> bf16 / fp16 -> global
#pragma unroll 1
      for (int t = 0; t <= t_last; ++t) {
        if (p.stats_tmem) {
          if (!w.wait(bar(L::bStats + t), (fs_par >> t) & 1, L::bStats + t, -1)) { ok = false; break; }
          fs_par ^= 1u << t;
        } else {
          if (!w.wait(bar(L::bCorrFull + t), (cf_par >> t) & 1, L::bCorrFull + t, -1)) { ok = false; break; }
          cf_par ^= 1u << t;
        }
        const float l = mail[t * kBlockM + r];
        mbar_arrive(bar(L::bCorrEmpty + t));
        if (!w.wait(bar(L::bOFinal + t), (of_par >> t) & 1, L::bOFinal + t, -1)) { ok = false; break; }
        of_par ^= 1u << t;
        tr.rec(kEvEpiStart + t, -1);
        tc_fence_after();
        const float inv = l > 0.f ? 1.f / l : 0.f;
        const int tile_pos0 = packed_pos(tk, t * kBlockM, p.gshift);   // sequence position of row 0
        const int tile_end = tile_pos0 + (kBlockM >> p.gshift);        // one past the tile's last position
        const uint32_t tO = tmem + lane_base + L::col_o(t);
        const bool full_tile = !p.part_out && tile_end <= tk.len && tk.tok0 + tile_end <= p.total_tokens;
        if (full_tile) {
          // Stage the tile in shared memory in the TMA's 128-byte-swizzled layout
          // (16-byte unit k of row r sits at unit k ^ (r % 8)), then one thread
          // stores it with the TMA ("Flash Attention 4", section "Tile Primitive 数据流":
          // O -> registers -> SMEM -> TMA store).
          if (!w.wait(bar(L::bOstFree), (ost_n & 1) ^ 1, L::bOstFree, -1)) { ok = false; break; }
          const uint32_t row_base = sOst + (uint32_t)r * 128u;
#pragma unroll 1
          for (int c = 0; c < D / 16; ++c) {
            uint32_t u[16];
            tmem_ld16(tO + c * 16, u);
            tmem_wait_ld();
            uint32_t pk[8];
#pragma unroll
            for (int e = 0; e < 8; ++e)
              pk[e] = pack_16x2<F16>(__uint_as_float(u[2 * e]) * inv, __uint_as_float(u[2 * e + 1]) * inv);
            const uint32_t slab = row_base + (uint32_t)(c >> 2) * L::kSlabBytes;
            const uint32_t k0 = (uint32_t)(c & 3) * 2;
            st_shared_v4(slab + (((k0 + 0) ^ (r & 7)) << 4), pk[0], pk[1], pk[2], pk[3]);
            st_shared_v4(slab + (((k0 + 1) ^ (r & 7)) << 4), pk[4], pk[5], pk[6], pk[7]);
          }
          fence_proxy_async_smem();
          mbar_arrive(bar(L::bOstReady));
          if (warp == 8) {
            if (!w.wait(bar(L::bOstReady), ost_n & 1, L::bOstReady, -1)) { ok = false; break; }
            if (lane == 0) {
#pragma unroll
              for (int c = 0; c < L::kHalves; ++c)
                tma_store_3d(&p.tm_o, sOst + c * L::kSlabBytes, c * 64, tk.kvh << p.gshift, tk.tok0 + tile_pos0);
              bulk_commit();
              bulk_wait_read_all();
              mbar_arrive(bar(L::bOstFree));
            }
            __syncwarp();
          }
          ++ost_n;
        } else if (p.part_out) {
          // one key range of a split task (or a key shard): normalised fp32 rows, merged later
          const int pos = tile_pos0 + (r >> p.gshift);
          const int head = (tk.kvh << p.gshift) + (r & ((1 << p.gshift) - 1));
          const bool valid = pos < tk.len && tk.tok0 + pos < p.total_tokens;
          float* orow = p.o_part + ((size_t)tk.split * p.total_tokens * p.H + (size_t)(tk.tok0 + pos) * p.H + head) * D;
#pragma unroll 1
          for (int c = 0; c < D / 16; ++c) {
            uint32_t u[16];
            tmem_ld16(tO + c * 16, u);
            tmem_wait_ld();
            if (valid) {
              float4* dst = reinterpret_cast<float4*>(orow + c * 16);
#pragma unroll
              for (int e = 0; e < 4; ++e)
                dst[e] = make_float4(__uint_as_float(u[4 * e]) * inv, __uint_as_float(u[4 * e + 1]) * inv,
                                     __uint_as_float(u[4 * e + 2]) * inv, __uint_as_float(u[4 * e + 3]) * inv);
            }
          }
        } else {
          // ragged tile: per-row stores, nothing past the sequence or the tensor
          const int pos = tile_pos0 + (r >> p.gshift);
          const int head = (tk.kvh << p.gshift) + (r & ((1 << p.gshift) - 1));
          const bool valid = pos < tk.len && tk.tok0 + pos < p.total_tokens;
          uint16_t* orow = p.o + ((size_t)(tk.tok0 + pos) * p.H + head) * D;
#pragma unroll 1
          for (int c = 0; c < D / 16; ++c) {
            uint32_t u[16];
            tmem_ld16(tO + c * 16, u);
            tmem_wait_ld();
            uint32_t pk[8];
#pragma unroll
            for (int e = 0; e < 8; ++e)
              pk[e] = pack_16x2<F16>(__uint_as_float(u[2 * e]) * inv, __uint_as_float(u[2 * e + 1]) * inv);
            if (valid) {
              uint4* dst = reinterpret_cast<uint4*>(orow + c * 16);
              dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
              dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
            }
          }
        }
        tr.rec(kEvEpiEnd + t, -1);
        tc_fence_before();
        mbar_arrive(bar(L::bPO + t));   // O_t is free for the next task's first PV
      }
    }
  }

  // the TMA stores of O must complete (and stop reading shared memory) before exit
  if (warp == 8 && lane == 0) bulk_wait_all();

  // ---- teardown: every role has returned; release tensor memory
  __syncwarp();  // lanes that skipped a single-thread role wait for lane 0
  tc_fence_before();
  __syncthreads();
  if (warp == 12) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace fa
