// fa_api.cu -- host side of the C ABI declared in include/fa.h: argument checks,
// TMA tensor maps, the varlen longest-first schedule kernel, kernel launches and
// the device status word.
#include <cuda.h>
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <functional>
#include <algorithm>
#include <queue>
#include <vector>
#include <array>
#include <map>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "fa.h"
#include "fa_fwd.cuh"
#include "fa_host.cuh"
#include "fa_selftest.h"

namespace {
using fa_host::aligned;
using fa_host::check_heads;
using fa_host::make_map;

// ------------------------------------------------------------------ options
struct Options {
  float tau = 8.0f;
  unsigned long long timeout_ns = 2000000000ull;
  int persistent = -1;   // -1: default (work stealing)
  int emu_groups = 0;
  int bwd_deterministic = 0;
  int stagger = 0;
  int stats_tmem = 1;
  int bwd_section = 0;
  int solo = -1;         // -1: the library's choice
};
Options g_opt;

// tracing builds: where fa_fwd / fa_fwd_varlen write their clock stamps
unsigned long long* g_trace_buf = nullptr;
int g_trace_ctas = 0;

// ------------------------------------------------------------------ per-device facts
struct DevInfo {
  bool init = false;
  bool supported = false;
  int sm_count = 0;
  long long l2_bytes = 0;
  bool attr_done[2][2][2][2][2] = {};   // [d == 128][causal][emulation][fp16][solo]
  int attr_status[2][2][2][2][2] = {};
};
constexpr int kMaxDevices = 64;
DevInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

int device_info(DevInfo** out) {
  int dev = 0;
  int n = 0;
  if (cudaGetDeviceCount(&n) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    return FA_ERR_NO_DEVICE;
  }
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DevInfo& d = g_dev[dev];
  if (!d.init) {
    int major = 0, minor = 0, sms = 0, l2 = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev) != cudaSuccess)
      return FA_ERR_CUDA;
    d.supported = (major == 10 && minor == 3);
    d.sm_count = sms;
    d.l2_bytes = l2;
    d.init = true;
  }
  *out = &d;
  return d.supported ? FA_OK : FA_ERR_UNSUPPORTED;
}

// The four maps of one call: Q and O ([tokens, H, d]) with H heads in boxes of G,
// K and V ([tokens_k, H_kv, d]) with H_kv heads.
int make_maps(fa::FwdParams& p, const void* q, const void* k, const void* v, void* o, long long tokens,
              long long tokens_k, int H, int Hkv, int d, bool f16) {
  const int G = H / Hkv;
  int st;
  if ((st = make_map(&p.tm_q, q, tokens, H, d, G, f16)) != FA_OK ||
      (st = make_map(&p.tm_k, k, tokens_k, Hkv, d, 1, f16)) != FA_OK ||
      (st = make_map(&p.tm_v, v, tokens_k, Hkv, d, 1, f16)) != FA_OK ||
      (st = make_map(&p.tm_o, o, tokens, H, d, G, f16)) != FA_OK)
    return st;
  return FA_OK;
}

// Key ranges per task. requested > 0: that many (at most one per 128-key block and
// kMaxSplits). requested = 0: the library's choice below.
constexpr int kMaxSplits = 128;
// Fixed length: split only when the unsplit tasks leave SMs idle. For each s up to 64
// the estimate runs the tasks through longest-first list scheduling on sm_count SMs,
// each task with its own key range (a causal task sees only the blocks up to its
// diagonal; the kernel cuts ranges of ceil(key_blocks / s) blocks, so a short causal
// task's upper ranges are empty) at (blocks * step + 2) for a range with keys and 1 for
// an empty one (it writes zero partials), in units of one two-tile K/V block step
// (about 2 us; a solo task's step, its QK^T overlapping the previous softmax, measures
// about 0.6 of it). The time is at least the unique K and V bytes at HBM speed (about
// 13 MB per unit). With s > 1 it adds the merge: its launch (2.5 units) and the fp32
// partials written and read back. A larger s must be at least 2 % faster to be taken.
// Decoding, 64 (sequence, K/V head) tasks over 256 key blocks on 152 SMs: two-tile
// tasks take 7 ranges (three rounds of 448 tasks, rather than 2 ranges leaving 24 SMs
// idle); solo tasks take 2 (one wave at the HBM floor: 164 against 168 us with 7).
// Cached per shape (a decoding loop asks every step).
int choose_splits_fixed(int requested, int B, int H, int H_kv, int num_m, int task_rows, int N_q, int N_kv, int d,
                        int gshift, bool causal, int sm_count) {
  const int key_blocks = (N_kv + fa::kBlockN - 1) / fa::kBlockN;
  const int most = key_blocks < 1 ? 1 : (key_blocks < kMaxSplits ? key_blocks : kMaxSplits);
  if (requested > 0) return requested < most ? requested : most;
  const long long base = (long long)B * H_kv * num_m;
  if (base >= sm_count || key_blocks < 2 || sm_count < 1) return 1;
  static std::mutex mu;
  static std::map<std::array<long long, 7>, int> cache;
  const std::array<long long, 7> key{B, (long long)H * 65536 + H_kv, (long long)num_m * 1024 + task_rows, N_q, N_kv,
                                     (long long)d * 64 + gshift * 2 + (causal ? 1 : 0), sm_count};
  {
    std::lock_guard<std::mutex> lk(mu);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
  }
  // each m's visible block count (the same for every (b, kv head))
  std::vector<int> nb(num_m);
  for (int m = 0; m < num_m; ++m) {
    long long kmax = N_kv;
    if (causal) {
      const long long last = ((long long)m * task_rows + task_rows - 1) >> gshift;
      kmax = std::min<long long>(last + (N_kv - N_q) + 1, N_kv);
    }
    nb[m] = kmax > 0 ? (int)((kmax + fa::kBlockN - 1) / fa::kBlockN) : 0;
  }
  const int limit = std::min(64, key_blocks);
  const double step = task_rows == fa::kBlockM ? 0.6 : 1.0;            // units per K/V block
  const double kv_floor = 4.0 * B * H_kv * (double)N_kv * d / 13e6;     // K and V once from HBM
  int best = 1;
  double best_time = -1.0;
  std::vector<double> costs;
  for (int sp = 1; sp <= limit; ++sp) {
    const int per = (key_blocks + sp - 1) / sp;
    costs.clear();
    for (long long bh = 0; bh < (long long)B * H_kv; ++bh)
      for (int m = 0; m < num_m; ++m)
        for (int r = 0; r < sp; ++r) {
          const int len = std::max(0, std::min(nb[m], (r + 1) * per) - r * per);
          costs.push_back(len > 0 ? len * step + 2.0 : 1.0);
        }
    std::sort(costs.begin(), costs.end(), std::greater<double>());
    std::priority_queue<double, std::vector<double>, std::greater<double>> load;
    for (int i = 0; i < sm_count; ++i) load.push(0.0);
    double makespan = 0.0;
    for (double c : costs) {
      const double t = load.top() + c;
      load.pop();
      load.push(t);
      makespan = std::max(makespan, t);
    }
    makespan = std::max(makespan, kv_floor);
    if (sp > 1) {
      const double partial_bytes = 2.0 * sp * (double)B * N_q * H * d * sizeof(float);
      makespan += 2.5 + partial_bytes / 13e6;
    }
    if (best_time < 0 || makespan < 0.98 * best_time) {
      best_time = makespan;
      best = sp;
    }
  }
  std::lock_guard<std::mutex> lk(mu);
  cache[key] = best;
  return best;
}

// Packed rows per fixed-length task: 256 (two Q tiles sharing each K/V block), or 128
// ("solo": one Q tile whose score tile alternates between S_0 and S_1, so that each
// block's QK^T overlaps the previous block's softmax) when the 256-row tasks leave SMs
// idle and the 128-row ones still fit in one wave (decoding, small batches).
int task_rows_fixed(int B, int H_kv, int N_q, int gshift, int sm_count) {
  if (g_opt.solo == 0 || g_opt.emu_groups > 0) return fa::kTaskRows;
  if (g_opt.solo == 1) return fa::kBlockM;
  const long long rows = (long long)N_q << gshift;
  const long long pairs = (long long)B * H_kv;
  const long long t256 = pairs * ((rows + fa::kTaskRows - 1) / fa::kTaskRows);
  const long long t128 = pairs * ((rows + fa::kBlockM - 1) / fa::kBlockM);
  return (t256 < sm_count && t128 <= sm_count) ? fa::kBlockM : fa::kTaskRows;
}

// Varlen: the same rule on an upper bound of the work tiles, H_kv * (ceil(total_q * G / rows)
// + num_seqs) (a sequence adds at most one partial tile).
long long varlen_tiles(long long total_q, int num_seqs, int H_kv, int gshift, int rows) {
  return (long long)H_kv * (((total_q << gshift) + rows - 1) / rows + num_seqs);
}
int task_rows_varlen(long long total_q, int num_seqs, int H_kv, int gshift, int sm_count) {
  if (g_opt.solo == 0 || g_opt.emu_groups > 0) return fa::kTaskRows;
  if (g_opt.solo == 1) return fa::kBlockM;
  return (varlen_tiles(total_q, num_seqs, H_kv, gshift, fa::kTaskRows) < sm_count &&
          varlen_tiles(total_q, num_seqs, H_kv, gshift, fa::kBlockM) <= sm_count)
             ? fa::kBlockM : fa::kTaskRows;
}

int choose_splits(int requested, long long base_tasks, int key_blocks, int sm_count) {
  const int most = key_blocks < 1 ? 1 : (key_blocks < kMaxSplits ? key_blocks : kMaxSplits);
  if (requested > 0) return requested < most ? requested : most;
  if (base_tasks >= sm_count || key_blocks < 8 || sm_count < 1) return 1;
  int limit = key_blocks / 4;
  if (limit > 64) limit = 64;
  int best = 1;
  long long best_cost = -1;
  for (int sp = 1; sp <= limit; ++sp) {
    const long long rounds = (base_tasks * sp + sm_count - 1) / sm_count;
    const long long cost = rounds * ((key_blocks + sp - 1) / sp + 2);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = sp;
    }
  }
  return best;
}

// Stream-ordered temporary buffer: `head_bytes` for the caller (the varlen tile
// list), then for splits > 0 the partial outputs o_part [splits][rows][d] fp32
// and lse_part [splits][rows] fp32.
struct Partials {
  void* base = nullptr;
  float* o_part = nullptr;
  float* lse_part = nullptr;
  int alloc(int splits, long long rows, int d, size_t head_bytes, cudaStream_t s) {
    const size_t o_bytes = splits > 0 ? (size_t)splits * (size_t)rows * d * sizeof(float) : 0;
    const size_t l_bytes = splits > 0 ? ((size_t)splits * (size_t)rows * sizeof(float) + 255) / 256 * 256 : 0;
    if (head_bytes + o_bytes + l_bytes == 0) return FA_OK;
    if (fa_host::alloc_async(&base, head_bytes + o_bytes + l_bytes, s) != cudaSuccess) {
      cudaGetLastError();
      base = nullptr;
      return FA_ERR_CUDA;
    }
    if (splits > 0) {
      o_part = reinterpret_cast<float*>(static_cast<char*>(base) + head_bytes);
      lse_part = reinterpret_cast<float*>(static_cast<char*>(base) + head_bytes + o_bytes);
    }
    return FA_OK;
  }
  int release(cudaStream_t s) {
    if (base == nullptr) return FA_OK;
    const bool ok = cudaFreeAsync(base, s) == cudaSuccess;
    base = nullptr;
    return ok ? FA_OK : FA_ERR_CUDA;
  }
};


template <int D, bool C, bool E, bool F, bool S>
int launch_fwd(DevInfo* dev, const fa::FwdParams& p, int grid, cudaStream_t stream) {
  using L = fa::Layout<D>;
  auto kern = fa::fa_fwd_kernel<D, C, E, F, S>;
  const int di = D == 128 ? 1 : 0, ci = C ? 1 : 0, ei = E ? 1 : 0, fi = F ? 1 : 0, si = S ? 1 : 0;
  {
    std::lock_guard<std::mutex> lk(g_dev_mu);
    if (!dev->attr_done[di][ci][ei][fi][si]) {
      int st = FA_OK;
      cudaFuncAttributes fa_attr;
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmemAlloc) != cudaSuccess ||
          cudaFuncGetAttributes(&fa_attr, kern) != cudaSuccess)
        st = FA_ERR_CUDA;
      // the warpgroup register split (192/192/48/80) needs exactly 128 registers
      // per thread at launch
      else if (fa_attr.numRegs != 128)
        st = FA_ERR_UNSUPPORTED;
      dev->attr_status[di][ci][ei][fi][si] = st;
      dev->attr_done[di][ci][ei][fi][si] = true;
    }
    if (dev->attr_status[di][ci][ei][fi][si] != FA_OK) return dev->attr_status[di][ci][ei][fi][si];
  }
  // A grid of one wave (latency-bound work) is launched with programmatic stream
  // serialization: its prologue (barriers, tensor memory, tensor-map prefetch) runs
  // while the previous kernel in the stream finishes, and it waits for that kernel
  // (griddepcontrol.wait) before touching global memory. Measured, CUDA graphs of 20
  // calls: B1 H1 N256 d64 6.95 -> 5.92 us, B2 H8 N1024 13.5 -> 13.15 us; larger grids
  // gained nothing (B4 H16 N4096 causal 0.9 % slower), so they keep the plain launch.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(fa::kThreads);
  cfg.dynamicSmemBytes = L::kSmemAlloc;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = grid <= dev->sm_count ? 1 : 0;
  fa::FwdParams q = p;
  q.pdl = cfg.numAttrs;
  if (cudaLaunchKernelEx(&cfg, kern, q) != cudaSuccess) return FA_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

// Solo tasks (task_rows 128) have their own kernel, without the polynomial exp2
// (task_rows_fixed keeps two-tile tasks when the emulation is on).
template <int D, bool C, bool F>
int dispatch_emu(DevInfo* dev, const fa::FwdParams& p, int grid, cudaStream_t s) {
  if (p.task_rows == fa::kBlockM) return launch_fwd<D, C, false, F, true>(dev, p, grid, s);
  return p.emu_groups > 0 ? launch_fwd<D, C, true, F, false>(dev, p, grid, s)
                          : launch_fwd<D, C, false, F, false>(dev, p, grid, s);
}

template <bool F>
int dispatch_t(DevInfo* dev, const fa::FwdParams& p, int d, bool causal, int grid, cudaStream_t s) {
  if (d == 128)
    return causal ? dispatch_emu<128, true, F>(dev, p, grid, s) : dispatch_emu<128, false, F>(dev, p, grid, s);
  return causal ? dispatch_emu<64, true, F>(dev, p, grid, s) : dispatch_emu<64, false, F>(dev, p, grid, s);
}

int dispatch(DevInfo* dev, const fa::FwdParams& p, int d, bool causal, bool f16, int grid, cudaStream_t s) {
  return f16 ? dispatch_t<true>(dev, p, d, causal, grid, s) : dispatch_t<false>(dev, p, d, causal, grid, s);
}

// fp16 weights P = 2^(s - ref) stay below 2^tau; fp16 holds up to 65504, so its
// threshold is capped at 15.
constexpr float kTauMaxF16 = 15.0f;

void fill_common(fa::FwdParams& p, float scale, bool f16) {
  p.sched = g_opt.persistent < 0 ? 2 : g_opt.persistent;
  p.trace = g_trace_buf;
  p.trace_ctas = g_trace_ctas;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.tau = f16 && g_opt.tau > kTauMaxF16 ? kTauMaxF16 : g_opt.tau;
  p.emu_groups = g_opt.emu_groups;
  p.stagger = g_opt.stagger;
  p.stats_tmem = g_opt.stats_tmem;
  p.timeout_ns = g_opt.timeout_ns;
}

// Grid size: one CTA per task, except the static-stride mode (one CTA per SM).
int grid_for(const fa::FwdParams& p, const DevInfo* dev, int n_tasks) {
  return (p.sched == 1 && n_tasks > dev->sm_count) ? dev->sm_count : n_tasks;
}

}  // namespace

// ------------------------------------------------------------------ varlen schedule kernel
namespace fa {
constexpr int kSchedBuckets = 4096;

// One CTA: enumerate the (sequence, rows-row block, key range) work tiles, bucket
// them by their number of K/V blocks, and write them longest first, each
// followed by all Hkv K/V heads ("FlashAttention-4（下）" (argus lesson 7),
// section "6. LPT 调度": sort work tiles by their cost, write a virtual -> actual
// map). Rows are packed (sequence position, query head of the group): a
// sequence of Lq query rows has Lq << gshift packed rows, and row r of a block
// sits at position r >> gshift. Tiles without keys (cost 0) are listed too: they
// write the rows' empty result.
//
// The offsets are checked first (the varlen design reads per-sequence offsets
// from cu_seqlens, "FlashAttention-4（下）" section "6. LPT 调度"): cu_q[0] =
// cu_k[0] = 0, both non-decreasing, and, where the argument is >= 0,
// cu_q[num_seqs] = total_q, cu_k[num_seqs] = total_k and every query length
// <= max_q. On a violation the kernel lists no tile (*count = 0, so the attention
// kernel and the merge write nothing) and records FA_ERR_INVALID_ARG | role 7 << 8 |
// (first offending index) << 32 in the device status word.
constexpr uint32_t kRoleSchedule = 7;
constexpr unsigned long long kStatusInvalid = 1;  // == FA_ERR_INVALID_ARG

__device__ __forceinline__ bool cu_entry_ok(const int* cu, int s, int num_seqs, int total, int max_len) {
  const int a = cu[s], b = cu[s + 1];
  if (b < a) return false;
  if (s == 0 && a != 0) return false;
  if (s == num_seqs - 1 && total >= 0 && b != total) return false;
  return max_len < 0 || b - a <= max_len;
}

__global__ void __launch_bounds__(1024) fa_varlen_schedule_kernel(const int* cu_q, const int* cu_k, int num_seqs,
                                                                  int Hkv, int gshift, int causal, int splits,
                                                                  int rows, int capacity, int4* tasks, int* count,
                                                                  int total_q, int total_k, int max_q,
                                                                  long long section_bytes, int kv_row_bytes) {
  griddep_launch_dependents();   // an attention grid of one wave may start its prologue now
  __shared__ int hist[kSchedBuckets];
  __shared__ int total_tiles;
  __shared__ int first_bad;
  __shared__ int max_cost;
  __shared__ long long sec_bytes;
  for (int i = threadIdx.x; i < kSchedBuckets; i += blockDim.x) hist[i] = 0;
  if (threadIdx.x == 0) {
    total_tiles = 0;
    first_bad = INT_MAX;
    max_cost = 0;
  }
  __syncthreads();
  for (int s = threadIdx.x; s < num_seqs; s += blockDim.x)
    if (!cu_entry_ok(cu_q, s, num_seqs, total_q, max_q) || !cu_entry_ok(cu_k, s, num_seqs, total_k, -1))
      atomicMin(&first_bad, s);
  __syncthreads();
  if (first_bad != INT_MAX) {
    if (threadIdx.x == 0) {
      *count = 0;
      atomicCAS(&g_fa_status, 0ull,
                kStatusInvalid | ((unsigned long long)kRoleSchedule << 8) |
                    ((unsigned long long)(uint32_t)first_bad << 32));
    }
    return;
  }
  auto cost_of = [&](int m, int Lq, int Lk, int sp) {
    const KRange r = key_range(m * rows, rows, Lk - Lq, Lk, gshift, causal != 0, splits, sp);
    return min(r.hi - r.lo, kSchedBuckets - 1);
  };
  // one warp per sequence, its lanes over the sequence's row blocks
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  int my_max = 0, my_tiles = 0;
  for (int s = warp; s < num_seqs; s += nwarps) {
    const int Lq = max(cu_q[s + 1] - cu_q[s], 0), Lk = max(cu_k[s + 1] - cu_k[s], 0);
    const int nm = ((Lq << gshift) + rows - 1) / rows;
    for (int m = lane; m < nm; m += 32)
      for (int sp = 0; sp < splits; ++sp) {
        my_max = max(my_max, cost_of(m, Lq, Lk, sp));
        ++my_tiles;
      }
  }
  atomicMax(&max_cost, my_max);
  atomicAdd(&total_tiles, my_tiles);
  __syncthreads();
  // L2 sections: consecutive sequences whose K and V (all K/V heads) fill about
  // section_bytes form one section (a sequence belongs to the section where its keys
  // start, so no scan is needed: cu_k is the prefix); the tiles are listed section by
  // section, longest first inside each, so the CTAs running at once share one
  // section's K/V in L2. Sort key = section * (max_cost + 1) + (max_cost - cost); the
  // sections grow until the keys fit in the histogram. section_bytes = 0: one section.
  const int nc = max_cost + 1;
  if (threadIdx.x == 0) {
    const long long all = (long long)total_k * kv_row_bytes;
    long long b = section_bytes > 0 ? section_bytes : all + 1;
    if (b < 1) b = 1;
    long long nsec = all / b + 1;
    if (nsec * nc > kSchedBuckets) {
      b *= (nsec * nc + kSchedBuckets - 1) / kSchedBuckets;
      nsec = all / b + 1;
      while (nsec * nc > kSchedBuckets) {   // integer rounding: grow until it fits
        b += b / 8 + 1;
        nsec = all / b + 1;
      }
    }
    sec_bytes = b;
  }
  __syncthreads();
  const long long sb = sec_bytes;
  auto key_of = [&](int s, int c) { return (int)(((long long)cu_k[s] * kv_row_bytes) / sb) * nc + (max_cost - c); };
  for (int s = warp; s < num_seqs; s += nwarps) {
    const int Lq = max(cu_q[s + 1] - cu_q[s], 0), Lk = max(cu_k[s + 1] - cu_k[s], 0);
    const int nm = ((Lq << gshift) + rows - 1) / rows;
    for (int m = lane; m < nm; m += 32)
      for (int sp = 0; sp < splits; ++sp) atomicAdd(&hist[key_of(s, cost_of(m, Lq, Lk, sp))], 1);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // exclusive scan in key order: hist[k] becomes the first slot of key k
    const long long all = (long long)total_k * kv_row_bytes;
    const int nkeys = (int)(all / sb + 1) * nc;
    int run = 0;
    for (int k = 0; k < nkeys; ++k) {
      const int n = hist[k];
      hist[k] = run;
      run += n;
    }
    const long long n_tasks = (long long)total_tiles * Hkv;
    *count = (int)(n_tasks < capacity ? n_tasks : capacity);
  }
  __syncthreads();
  for (int s = warp; s < num_seqs; s += nwarps) {
    const int Lq = max(cu_q[s + 1] - cu_q[s], 0), Lk = max(cu_k[s + 1] - cu_k[s], 0);
    const int nm = ((Lq << gshift) + rows - 1) / rows;
    for (int m = lane; m < nm; m += 32) {
      for (int sp = 0; sp < splits; ++sp) {
        const int c = cost_of(m, Lq, Lk, sp);
        const int slot = atomicAdd(&hist[key_of(s, c)], 1);
        for (int h = 0; h < Hkv; ++h) {
          const long long ti = (long long)slot * Hkv + h;
          if (ti < capacity) tasks[ti] = make_int4(s, h | (sp << 16), m, c);
        }
      }
    }
  }
}

// Merge of partial results over disjoint key ranges, one warp per (row, head):
//   LSE = ln sum_s exp(LSE_s),  O = sum_s exp(LSE_s - LSE) O_s
// parts with LSE_s = -inf are skipped (their O_s is not read); a row without
// any key gets O = 0, LSE = -inf. ("FlashAttention：一次前向计算", the two-round
// example: partial results over key blocks are brought to one reference and
// divided once by the total denominator; "Flash Attention 4", section
// "重缩放与结果写回": the LSE of each part.)
// o_part [parts][rows][H][D] fp32 (normalised per part); lse_part [parts][...]:
// the LSE of (row, head) sits at ((row / nl) * H + head) * nl + row % nl.
template <int D, bool F16>
__global__ void __launch_bounds__(256) fa_combine_kernel(const float* __restrict__ o_part,
                                                         const float* __restrict__ lse_part, int parts,
                                                         long long o_stride, long long lse_stride, int rows, int H,
                                                         int nl, uint16_t* __restrict__ o, float* __restrict__ lse,
                                                         const int* __restrict__ task_count) {
  // a varlen call whose schedule kernel rejected cu_seqlens listed no tile: write nothing
  if (task_count != nullptr && *task_count == 0) return;
  constexpr int E = D / 32;   // floats per lane
  const long long w = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (w >= (long long)rows * H) return;
  const int lane = threadIdx.x & 31;
  const int row = (int)(w / H), h = (int)(w % H);
  const long long li = ((long long)(row / nl) * H + h) * nl + row % nl;
  float m = -INFINITY;
  for (int s = lane; s < parts; s += 32) m = fmaxf(m, lse_part[s * lse_stride + li]);
#pragma unroll
  for (int x = 16; x > 0; x >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, x));
  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  float sum = 0.f;
  if (m != -INFINITY) {
    for (int s = 0; s < parts; ++s) {
      const float l = lse_part[s * lse_stride + li];
      if (l == -INFINITY) continue;
      const float wgt = ex2_approx((l - m) * 1.4426950408889634f);
      sum += wgt;
      const float* src = o_part + s * o_stride + w * D + lane * E;
      if constexpr (E == 4) {
        const float4 x = *reinterpret_cast<const float4*>(src);
        acc[0] += wgt * x.x; acc[1] += wgt * x.y; acc[2] += wgt * x.z; acc[3] += wgt * x.w;
      } else {
        const float2 x = *reinterpret_cast<const float2*>(src);
        acc[0] += wgt * x.x; acc[1] += wgt * x.y;
      }
    }
  }
  const float inv = sum > 0.f ? 1.f / sum : 0.f;
  uint32_t* dst = reinterpret_cast<uint32_t*>(o + w * D + lane * E);
#pragma unroll
  for (int e = 0; e < E; e += 2) dst[e / 2] = pack_16x2<F16>(acc[e] * inv, acc[e + 1] * inv);
  if (lse != nullptr && lane == 0)
    lse[li] = m == -INFINITY ? -INFINITY : m + lg2_approx(sum) * 0.69314718055994531f;
}
}  // namespace fa

namespace {
int launch_combine(const float* o_part, const float* lse_part, int parts, long long o_stride, long long lse_stride,
                   int rows, int H, int nl, int d, bool f16, void* o, float* lse, cudaStream_t s,
                   const int* task_count = nullptr) {
  const long long warps = (long long)rows * H;
  const long long blocks = (warps + 7) / 8;
  if (blocks > INT_MAX) return FA_ERR_INVALID_ARG;
  uint16_t* out = static_cast<uint16_t*>(o);
  const int g = (int)blocks;
  if (d == 128) {
    if (f16) fa::fa_combine_kernel<128, true><<<g, 256, 0, s>>>(o_part, lse_part, parts, o_stride, lse_stride, rows, H, nl, out, lse, task_count);
    else fa::fa_combine_kernel<128, false><<<g, 256, 0, s>>>(o_part, lse_part, parts, o_stride, lse_stride, rows, H, nl, out, lse, task_count);
  } else {
    if (f16) fa::fa_combine_kernel<64, true><<<g, 256, 0, s>>>(o_part, lse_part, parts, o_stride, lse_stride, rows, H, nl, out, lse, task_count);
    else fa::fa_combine_kernel<64, false><<<g, 256, 0, s>>>(o_part, lse_part, parts, o_stride, lse_stride, rows, H, nl, out, lse, task_count);
  }
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}
}  // namespace

// ------------------------------------------------------------------ fixed-length parameters
namespace {
// Argument checks and kernel parameters of a fixed-length call (everything but the
// outputs): maps of q, k, v and o (o only for the TMA store of full 16-bit tiles),
// task shape and count, key splits, L2 sections.
int fixed_params(fa::FwdParams& p, DevInfo** devp, const void* q, const void* k, const void* v, const void* o,
                 int B, int H, int H_kv, int N_q, int N_kv, int d, float scale, int causal, int dtype,
                 int num_splits) {
  if (!q || !k || !v) return FA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16)) return FA_ERR_INVALID_ARG;
  if (B <= 0 || H <= 0 || H_kv <= 0 || N_q <= 0 || N_kv <= 0 || num_splits < 0) return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  if (dtype != FA_DTYPE_BF16 && dtype != FA_DTYPE_FP16) return FA_ERR_INVALID_ARG;
  int gshift = 0;
  int st = check_heads(H, H_kv, &gshift);
  if (st != FA_OK) return st;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  const long long tokens = (long long)B * N_q, tokens_k = (long long)B * N_kv;
  if (tokens * H > INT_MAX || tokens_k * H_kv > INT_MAX) return FA_ERR_INVALID_ARG;  // 32-bit row indexing
  DevInfo* dev = nullptr;
  if ((st = device_info(&dev)) != FA_OK) return st;
  *devp = dev;
  const bool f16 = dtype == FA_DTYPE_FP16;
  std::memset(&p, 0, sizeof p);
  if ((st = make_maps(p, q, k, v, const_cast<void*>(o), tokens, tokens_k, H, H_kv, d, f16)) != FA_OK) return st;
  p.B = B; p.H = H; p.N = N_q; p.Nk = N_kv;
  p.Hkv = H_kv;
  p.gshift = gshift;
  p.total_tokens = (int)tokens;
  // tasks of task_rows packed rows; a (b, kv head) has N_q * G rows
  p.task_rows = task_rows_fixed(B, H_kv, N_q, gshift, dev->sm_count);
  p.num_m = (int)((((long long)N_q << gshift) + p.task_rows - 1) / p.task_rows);
  const long long base_tasks = (long long)B * H_kv * p.num_m;
  p.splits = choose_splits_fixed(num_splits, B, H, H_kv, p.num_m, p.task_rows, N_q, N_kv, d, gshift, causal != 0,
                                 dev->sm_count);
  const long long ntask = base_tasks * p.splits;
  if (ntask > INT_MAX) return FA_ERR_INVALID_ARG;
  p.num_tasks = (int)ntask;
  // L2 sections of (b, kv head) pairs whose K + V fill a quarter of L2: measured on
  // B4 H16 N4096 (201.7 -> 199.2 us per call) and grouped B4 H32/8 N4096 (387.7 ->
  // 385.7) against half of L2; an eighth or less is slower (fewer pairs to balance
  // the longest-first order over), larger sections too (c3 204 us with one section)
  const long long kv_bytes = 4LL * N_kv * d;                    // K + V of one (b, kv head)
  long long group = (dev->l2_bytes / 4) / (kv_bytes > 0 ? kv_bytes : 1);
  if (group < 1) group = 1;
  if (group > (long long)B * H_kv) group = (long long)B * H_kv;
  p.lpt_group = (int)group;
  p.varlen = 0;
  fill_common(p, scale, f16);
  return FA_OK;
}
}  // namespace

// ------------------------------------------------------------------ allocation-free scratch
namespace {
// Scratch of fa_fwd_varlen_noalloc: kNoAllocMaxTasks work tiles (int4 each)
// followed by one int4 whose first word is the tile count. A file-scope device
// array, so it exists on every GPU that loads this library until the process
// exits. Host code must not use the symbol as an address: noalloc_scratch()
// looks the device address up (once per device, with that device current).
constexpr int kNoAllocMaxTasks = 1 << 17;
static __device__ __align__(256) int4 g_noalloc_scratch[kNoAllocMaxTasks + 1];
int4* g_noalloc_ptr[kMaxDevices] = {};

int noalloc_scratch(int4** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) {
      cudaGetLastError();
      return FA_ERR_CUDA;
    }
    g_noalloc_ptr[dev] = static_cast<int4*>(ptr);
  }
  *out = g_noalloc_ptr[dev];
  return FA_OK;
}
}  // namespace

namespace fa_host {
void trace_target(unsigned long long** buf, int* ctas) {
  *buf = g_trace_buf;
  *ctas = g_trace_ctas;
}
bool bwd_deterministic() { return g_opt.bwd_deterministic != 0; }
int bwd_section_override() { return g_opt.bwd_section; }
int persistent_mode() { return g_opt.persistent; }
unsigned long long wait_timeout_ns() { return g_opt.timeout_ns; }

// The library's stream-ordered memory pool on the current device: unlike the default
// pool (release threshold 0, so its memory goes back to the system at every
// synchronisation and the next call maps it again, ~100 us), it keeps what it has
// allocated for the next call.
std::mutex g_pool_mu;
cudaMemPool_t g_pools[kMaxDevices] = {};

cudaError_t alloc_async(void** ptr, size_t bytes, cudaStream_t s) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  cudaMemPool_t pool = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_pool_mu);
    if (g_pools[dev] == nullptr) {
      cudaMemPoolProps props;
      std::memset(&props, 0, sizeof props);
      props.allocType = cudaMemAllocationTypePinned;
      props.handleTypes = cudaMemHandleTypeNone;
      props.location.type = cudaMemLocationTypeDevice;
      props.location.id = dev;
      cudaMemPool_t created = nullptr;
      if ((e = cudaMemPoolCreate(&created, &props)) != cudaSuccess) return e;
      uint64_t keep = UINT64_MAX;
      if ((e = cudaMemPoolSetAttribute(created, cudaMemPoolAttrReleaseThreshold, &keep)) != cudaSuccess) {
        cudaMemPoolDestroy(created);
        return e;
      }
      g_pools[dev] = created;
    }
    pool = g_pools[dev];
  }
  return cudaMallocFromPoolAsync(ptr, bytes, pool, s);
}

cudaError_t release_pools() {
  std::lock_guard<std::mutex> lk(g_pool_mu);
  for (cudaMemPool_t pool : g_pools)
    if (pool != nullptr) {
      const cudaError_t e = cudaMemPoolTrimTo(pool, 0);
      if (e != cudaSuccess) return e;
    }
  return cudaSuccess;
}
}  // namespace fa_host

// ------------------------------------------------------------------ C ABI
extern "C" {

int fa_version(void) { return 100; }

int fa_release_cached_memory(void) {
  if (fa_host::release_pools() != cudaSuccess) {
    cudaGetLastError();
    return FA_ERR_CUDA;
  }
  return FA_OK;
}

const char* fa_error_string(int status) {
  switch (status) {
    case FA_OK: return "ok";
    case FA_ERR_INVALID_ARG: return "invalid argument";
    case FA_ERR_UNSUPPORTED: return "unsupported (head dim, device or kernel resources)";
    case FA_ERR_CUDA: return "CUDA runtime/driver error";
    case FA_ERR_TIMEOUT: return "device-side wait timed out";
    case FA_ERR_NO_DEVICE: return "no CUDA device";
    case FA_ERR_CAPACITY: return "problem larger than the fixed scratch of the allocation-free entry point";
    default: return "unknown status";
  }
}

int fa_set_option(int option, double value) {
  switch (option) {
    case FA_OPT_TAU:
      if (!(value >= 0.0)) return FA_ERR_INVALID_ARG;  // also rejects NaN
      g_opt.tau = value > 3.0e38 ? INFINITY : (float)value;
      return FA_OK;
    case FA_OPT_WAIT_TIMEOUT_NS:
      if (!(value >= 1000.0 && value <= 6.0e11)) return FA_ERR_INVALID_ARG;
      g_opt.timeout_ns = (unsigned long long)value;
      return FA_OK;
    case FA_OPT_PERSISTENT:
      if (value != -1.0 && value != 0.0 && value != 1.0 && value != 2.0) return FA_ERR_INVALID_ARG;
      g_opt.persistent = (int)value;
      return FA_OK;
    case FA_OPT_EXP2_EMULATION:
      if (!(value >= 0.0 && value <= 8.0) || value != std::floor(value)) return FA_ERR_INVALID_ARG;
      g_opt.emu_groups = (int)value;
      return FA_OK;
    case FA_OPT_BWD_DETERMINISTIC:
      if (value != 0.0 && value != 1.0) return FA_ERR_INVALID_ARG;
      g_opt.bwd_deterministic = (int)value;
      return FA_OK;
    case FA_OPT_SOFTMAX_STAGGER:
      if (value != 0.0 && value != 1.0) return FA_ERR_INVALID_ARG;
      g_opt.stagger = (int)value;
      return FA_OK;
    case FA_OPT_STATS_TMEM:
      if (value != 0.0 && value != 1.0) return FA_ERR_INVALID_ARG;
      g_opt.stats_tmem = (int)value;
      return FA_OK;
    case FA_OPT_BWD_SECTION:
      if (!(value >= 0.0 && value <= 1e6) || value != std::floor(value)) return FA_ERR_INVALID_ARG;
      g_opt.bwd_section = (int)value;
      return FA_OK;
    case FA_OPT_SOLO_TILES:
      if (value != -1.0 && value != 0.0 && value != 1.0) return FA_ERR_INVALID_ARG;
      g_opt.solo = (int)value;
      return FA_OK;
    default:
      return FA_ERR_INVALID_ARG;
  }
}

int fa_fwd_kv(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int H_kv, int N_q,
              int N_kv, int d, float scale, int causal, int dtype, int num_splits, void* stream) {
  if (!o || !aligned(o, 16) || (lse && !aligned(lse, 4))) return FA_ERR_INVALID_ARG;
  fa::FwdParams p;
  DevInfo* dev = nullptr;
  int st = fixed_params(p, &dev, q, k, v, o, B, H, H_kv, N_q, N_kv, d, scale, causal, dtype, num_splits);
  if (st != FA_OK) return st;
  p.o = static_cast<uint16_t*>(o);
  p.lse = lse;
  const bool f16 = dtype == FA_DTYPE_FP16;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int grid = grid_for(p, dev, p.num_tasks);
  if (p.splits == 1) return dispatch(dev, p, d, causal != 0, f16, grid, s);

  // split keys: partial results in a temporary buffer, then the merge
  const long long tokens = (long long)B * N_q;
  Partials ws;
  if ((st = ws.alloc(p.splits, tokens * H, d, 0, s)) != FA_OK) return st;
  p.part_out = 1;
  p.o_part = ws.o_part;
  p.lse_part = ws.lse_part;
  p.lse_split_stride = tokens * H;
  st = dispatch(dev, p, d, causal != 0, f16, grid, s);
  if (st == FA_OK)
    st = launch_combine(ws.o_part, ws.lse_part, p.splits, tokens * H * d, tokens * H, (int)tokens, H, N_q, d, f16,
                        o, lse, s);
  const int fst = ws.release(s);
  return st != FA_OK ? st : fst;
}

int fa_fwd_kv_partial(const void* q, const void* k, const void* v, float* o_part, float* lse_part, int B, int H,
                      int H_kv, int N_q, int N_kv, int N_kv_total, int kv_offset, int d, float scale, int causal,
                      int dtype, void* stream) {
  if (!o_part || !lse_part || !aligned(o_part, 16) || !aligned(lse_part, 4)) return FA_ERR_INVALID_ARG;
  if (N_kv <= 0 || kv_offset < 0 || N_kv_total < N_kv || (long long)kv_offset + N_kv > N_kv_total)
    return FA_ERR_INVALID_ARG;
  fa::FwdParams p;
  DevInfo* dev = nullptr;
  // The O tensor map is built over q and never used: partial rows are written as fp32
  // by per-row stores, not by the TMA store of 16-bit tiles.
  int st = fixed_params(p, &dev, q, k, v, q, B, H, H_kv, N_q, N_kv, d, scale, causal, dtype, 1);
  if (st != FA_OK) return st;
  p.part_out = 1;
  p.o_part = o_part;
  p.lse_part = lse_part;
  p.lse_split_stride = 0;
  p.diag_shift = N_kv_total - kv_offset - N_kv;   // keys of the sequence after this shard
  const bool f16 = dtype == FA_DTYPE_FP16;
  return dispatch(dev, p, d, causal != 0, f16, grid_for(p, dev, p.num_tasks), static_cast<cudaStream_t>(stream));
}

int fa_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int H_kv, int N,
               int d, float scale, int causal, int dtype, void* stream) {
  return fa_fwd_kv(q, k, v, o, lse, B, H, H_kv, N, N, d, scale, causal, dtype, 1, stream);
}

int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
           float scale, int causal, void* stream) {
  return fa_fwd_gqa(q, k, v, o, lse, B, H, H, N, d, scale, causal, FA_DTYPE_BF16, stream);
}

}  // extern "C"

namespace {
// Argument checks shared by the varlen entry points; *cap = the task-list
// capacity: H_kv * (ceil(T * G / 256) + num_seqs) tiles of 256 packed rows, per key range.
int varlen_check(const void* q, const void* k, const void* v, void* o, float* lse, const int* cu_q, const int* cu_k,
                 int num_seqs, int total_q, int total_k, int max_q, int max_k, int H, int H_kv, int d, float scale,
                 int causal, int dtype, int num_splits, int* gshift, long long* base) {
  if (!q || !k || !v || !o || !cu_q || !cu_k) return FA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || (lse && !aligned(lse, 4)) ||
      !aligned(cu_q, 4) || !aligned(cu_k, 4))
    return FA_ERR_INVALID_ARG;
  if (num_seqs <= 0 || total_q <= 0 || total_k <= 0 || max_q <= 0 || max_k < 0 || H <= 0 || H_kv <= 0 ||
      num_splits < 0)
    return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  if (dtype != FA_DTYPE_BF16 && dtype != FA_DTYPE_FP16) return FA_ERR_INVALID_ARG;
  int st = check_heads(H, H_kv, gshift);
  if (st != FA_OK) return st;
  if (H_kv > 0xffff) return FA_ERR_UNSUPPORTED;   // the task list keeps the K/V head in 16 bits
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if ((long long)total_q * H > INT_MAX || (long long)total_k * H_kv > INT_MAX) return FA_ERR_INVALID_ARG;
  *base = (long long)H_kv * ((((long long)total_q << *gshift) + fa::kTaskRows - 1) / fa::kTaskRows + num_seqs);
  return FA_OK;
}

// Maps, schedule kernel, attention kernel (and with splits > 1 the merge) of a
// varlen call whose task list lives in tasks[0, cap) with its count at *count.
int varlen_launch(DevInfo* dev, const void* q, const void* k, const void* v, void* o, float* lse, const int* cu_q,
                  const int* cu_k, int num_seqs, int total_q, int total_k, int max_q, int H, int H_kv, int gshift, int d,
                  float scale, int causal, bool f16, int splits, int rows, const Partials* parts, int4* tasks,
                  int* count, int cap, cudaStream_t s) {
  fa::FwdParams p;
  std::memset(&p, 0, sizeof p);
  int st = make_maps(p, q, k, v, o, total_q, total_k, H, H_kv, d, f16);
  if (st != FA_OK) return st;
  // L2 sections of a quarter of L2 of K/V, as for fixed-length causal work
  fa::fa_varlen_schedule_kernel<<<1, 1024, 0, s>>>(cu_q, cu_k, num_seqs, H_kv, gshift, causal, splits, rows, cap,
                                                   tasks, count, total_q, total_k, max_q, dev->l2_bytes / 4,
                                                   H_kv * 4 * d);
  if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
  p.o = static_cast<uint16_t*>(o);
  p.lse = lse;
  p.cu_seqlens = cu_q;
  p.cu_seqlens_k = cu_k;
  p.tasks = tasks;
  p.task_count = count;
  p.H = H;
  p.Hkv = H_kv;
  p.gshift = gshift;
  p.total_tokens = total_q;
  p.num_tasks = cap;
  p.varlen = 1;
  p.task_rows = rows;
  p.splits = splits;
  if (splits > 1) {
    p.part_out = 1;
    p.o_part = parts->o_part;
    p.lse_part = parts->lse_part;
    p.lse_split_stride = (long long)total_q * H;
  }
  fill_common(p, scale, f16);
  const int grid = grid_for(p, dev, cap);
  st = dispatch(dev, p, d, causal != 0, f16, grid, s);
  if (st != FA_OK || splits == 1) return st;
  return launch_combine(parts->o_part, parts->lse_part, splits, (long long)total_q * H * d, (long long)total_q * H,
                        total_q, H, total_q, d, f16, o, lse, s, count);
}
}  // namespace

extern "C" {

int fa_fwd_varlen_kv(const void* q, const void* k, const void* v, void* o, float* lse, const int* cu_seqlens_q,
                     const int* cu_seqlens_kv, int num_seqs, int total_q, int total_kv, int max_seqlen_q,
                     int max_seqlen_kv, int H, int H_kv, int d, float scale, int causal, int dtype, int num_splits,
                     void* stream) {
  int gshift = 0;
  long long base = 0;
  int st = varlen_check(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_kv, num_seqs, total_q, total_kv, max_seqlen_q,
                        max_seqlen_kv, H, H_kv, d, scale, causal, dtype, num_splits, &gshift, &base);
  if (st != FA_OK) return st;
  DevInfo* dev = nullptr;
  if ((st = device_info(&dev)) != FA_OK) return st;
  const int rows = task_rows_varlen(total_q, num_seqs, H_kv, gshift, dev->sm_count);
  base = varlen_tiles(total_q, num_seqs, H_kv, gshift, rows);
  const int splits = choose_splits(num_splits, base, (max_seqlen_kv + fa::kBlockN - 1) / fa::kBlockN,
                                   dev->sm_count);
  const long long cap = base * splits;
  if (cap > INT_MAX) return FA_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool f16 = dtype == FA_DTYPE_FP16;
  // one temporary buffer: the tile list, its count, and with splits the partial results
  Partials ws;
  const size_t list_bytes = ((size_t)cap * sizeof(int4) + 16 + 255) / 256 * 256;
  if ((st = ws.alloc(splits > 1 ? splits : 0, (long long)total_q * H, d, list_bytes, s)) != FA_OK) return st;
  int4* tasks = static_cast<int4*>(ws.base);
  int* count = reinterpret_cast<int*>(static_cast<char*>(ws.base) + (size_t)cap * sizeof(int4));
  st = varlen_launch(dev, q, k, v, o, lse, cu_seqlens_q, cu_seqlens_kv, num_seqs, total_q, total_kv, max_seqlen_q,
                     H, H_kv, gshift,
                     d, scale, causal, f16, splits, rows, &ws, tasks, count, (int)cap, s);
  const int fst = ws.release(s);
  return st != FA_OK ? st : fst;
}

int fa_fwd_varlen_gqa(const void* q, const void* k, const void* v, void* o, float* lse, const int* cu_seqlens,
                      int num_seqs, int total_tokens, int max_seqlen, int H, int H_kv, int d, float scale,
                      int causal, int dtype, void* stream) {
  return fa_fwd_varlen_kv(q, k, v, o, lse, cu_seqlens, cu_seqlens, num_seqs, total_tokens, total_tokens, max_seqlen,
                          max_seqlen, H, H_kv, d, scale, causal, dtype, 1, stream);
}

int fa_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse, const int* cu_seqlens,
                  int num_seqs, int total_tokens, int max_seqlen, int H, int d, float scale, int causal,
                  void* stream) {
  return fa_fwd_varlen_gqa(q, k, v, o, lse, cu_seqlens, num_seqs, total_tokens, max_seqlen, H, H, d, scale, causal,
                           FA_DTYPE_BF16, stream);
}

int fa_fwd_kv_splits(int B, int H, int H_kv, int N_q, int N_kv, int d, int causal, int num_splits, int* splits) {
  if (!splits || B <= 0 || H <= 0 || H_kv <= 0 || N_q <= 0 || N_kv <= 0 || num_splits < 0) return FA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  int gshift = 0;
  int st = check_heads(H, H_kv, &gshift);
  if (st != FA_OK) return st;
  DevInfo* dev = nullptr;
  if ((st = device_info(&dev)) != FA_OK) return st;
  const int task_rows = task_rows_fixed(B, H_kv, N_q, gshift, dev->sm_count);
  const long long num_m = (((long long)N_q << gshift) + task_rows - 1) / task_rows;
  if ((long long)B * H_kv * num_m > INT_MAX) return FA_ERR_INVALID_ARG;
  *splits = choose_splits_fixed(num_splits, B, H, H_kv, (int)num_m, task_rows, N_q, N_kv, d, gshift, causal != 0,
                                dev->sm_count);
  return FA_OK;
}

int fa_fwd_varlen_kv_splits(int num_seqs, int total_q, int max_seqlen_kv, int H, int H_kv, int num_splits,
                            int* splits) {
  if (!splits || num_seqs <= 0 || total_q <= 0 || max_seqlen_kv < 0 || H <= 0 || H_kv <= 0 || num_splits < 0)
    return FA_ERR_INVALID_ARG;
  int gshift = 0;
  int st = check_heads(H, H_kv, &gshift);
  if (st != FA_OK) return st;
  DevInfo* dev = nullptr;
  if ((st = device_info(&dev)) != FA_OK) return st;
  const long long base =
      varlen_tiles(total_q, num_seqs, H_kv, gshift, task_rows_varlen(total_q, num_seqs, H_kv, gshift, dev->sm_count));
  *splits = choose_splits(num_splits, base, (max_seqlen_kv + fa::kBlockN - 1) / fa::kBlockN, dev->sm_count);
  return FA_OK;
}

int fa_lse_combine(const float* o_parts, const float* lse_parts, int num_parts, int B, int N, int H, int d, void* o,
                   float* lse, int dtype, void* stream) {
  if (!o_parts || !lse_parts || !o) return FA_ERR_INVALID_ARG;
  if (!aligned(o_parts, 16) || !aligned(lse_parts, 4) || !aligned(o, 16) || (lse && !aligned(lse, 4)))
    return FA_ERR_INVALID_ARG;
  if (num_parts <= 0 || B <= 0 || N <= 0 || H <= 0) return FA_ERR_INVALID_ARG;
  if (dtype != FA_DTYPE_BF16 && dtype != FA_DTYPE_FP16) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  const long long rows = (long long)B * N;
  if (rows > INT_MAX || rows * H > INT_MAX) return FA_ERR_INVALID_ARG;
  DevInfo* dev = nullptr;
  int st = device_info(&dev);
  if (st != FA_OK) return st;
  return launch_combine(o_parts, lse_parts, num_parts, rows * H * d, rows * H, (int)rows, H, N, d,
                        dtype == FA_DTYPE_FP16, o, lse, static_cast<cudaStream_t>(stream));
}

int fa_trace_configure(void* buf, int ctas) {
#ifdef FA_TRACE
  if (ctas < 0 || (ctas > 0 && (buf == nullptr || !aligned(buf, 8)))) return FA_ERR_INVALID_ARG;
  g_trace_buf = ctas > 0 ? static_cast<unsigned long long*>(buf) : nullptr;
  g_trace_ctas = ctas;
  return FA_OK;
#else
  (void)buf;
  (void)ctas;
  return FA_ERR_UNSUPPORTED;
#endif
}

int fa_trace_layout(int* roles, int* slots_per_role) {
  if (!roles || !slots_per_role) return FA_ERR_INVALID_ARG;
  *roles = fa::kTraceRoles;
  *slots_per_role = fa::kTraceSlots;
  return FA_OK;
}

int fa_varlen_schedule(const int* cu_seqlens_q, const int* cu_seqlens_kv, int num_seqs, int H_kv, int group,
                       int causal, int splits, int capacity, void* tasks, int* count, void* stream) {
  if (!cu_seqlens_q || !cu_seqlens_kv || !tasks || !count || num_seqs <= 0 || H_kv <= 0 || H_kv > 0xffff ||
      capacity < 0 || splits <= 0 || splits > kMaxSplits || (causal != 0 && causal != 1))
    return FA_ERR_INVALID_ARG;
  if (!aligned(tasks, 16) || !aligned(count, 4) || !aligned(cu_seqlens_q, 4) || !aligned(cu_seqlens_kv, 4))
    return FA_ERR_INVALID_ARG;
  int gshift = 0;
  if (group <= 0) return FA_ERR_INVALID_ARG;
  int st = check_heads(H_kv * group, H_kv, &gshift);
  if (st != FA_OK) return st;
  DevInfo* dev = nullptr;
  if ((st = device_info(&dev)) != FA_OK) return st;
  fa::fa_varlen_schedule_kernel<<<1, 1024, 0, static_cast<cudaStream_t>(stream)>>>(
      cu_seqlens_q, cu_seqlens_kv, num_seqs, H_kv, gshift, causal, splits, fa::kTaskRows, capacity,
      static_cast<int4*>(tasks), count, -1, -1, -1, 0, 0);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int fa_fwd_varlen_noalloc(const void* q, const void* k, const void* v, void* o, float* lse, const int* cu_seqlens,
                          int num_seqs, int total_tokens, int max_seqlen, int H, int d, float scale, int causal,
                          void* stream) {
  int gshift = 0;
  long long cap = 0;
  int st = varlen_check(q, k, v, o, lse, cu_seqlens, cu_seqlens, num_seqs, total_tokens, total_tokens, max_seqlen,
                        max_seqlen, H, H, d, scale, causal, FA_DTYPE_BF16, 1, &gshift, &cap);
  if (st != FA_OK) return st;
  // Refuse before touching the device when the tile bound of 256-row tasks, or of 128-row
  // tasks if FA_OPT_SOLO_TILES forces them, is already too large for the array.
  if (cap > kNoAllocMaxTasks) return FA_ERR_CAPACITY;
  if (g_opt.solo == 1 && varlen_tiles(total_tokens, num_seqs, H, gshift, fa::kBlockM) > kNoAllocMaxTasks)
    return FA_ERR_CAPACITY;
  DevInfo* dev = nullptr;
  if ((st = device_info(&dev)) != FA_OK) return st;
  // The schedule kernel writes up to `cap` tiles: check the bound of the row count chosen.
  const int rows = task_rows_varlen(total_tokens, num_seqs, H, gshift, dev->sm_count);
  cap = varlen_tiles(total_tokens, num_seqs, H, gshift, rows);
  if (cap > kNoAllocMaxTasks) return FA_ERR_CAPACITY;
  int4* scratch = nullptr;
  if ((st = noalloc_scratch(&scratch)) != FA_OK) return st;
  int4* tasks = scratch;
  int* count = reinterpret_cast<int*>(scratch + kNoAllocMaxTasks);
  return varlen_launch(dev, q, k, v, o, lse, cu_seqlens, cu_seqlens, num_seqs, total_tokens, total_tokens,
                       max_seqlen, H, H,
                       gshift, d, scale, causal, false, 1, rows, nullptr, tasks, count, (int)cap,
                       static_cast<cudaStream_t>(stream));
}

int fa_last_device_status(void* stream, unsigned long long* detail) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return FA_ERR_CUDA;
  unsigned long long word = 0, bwd_word = 0;
  if (cudaMemcpyFromSymbol(&word, fa::g_fa_status, sizeof word) != cudaSuccess) return FA_ERR_CUDA;
  if (word != 0) {
    const unsigned long long zero = 0;
    if (cudaMemcpyToSymbol(fa::g_fa_status, &zero, sizeof zero) != cudaSuccess) return FA_ERR_CUDA;
  }
  if (fa_host::bwd_take_status(&bwd_word) != FA_OK) return FA_ERR_CUDA;
  if (word == 0) word = bwd_word;
  if (detail) *detail = word;
  return word != 0 ? (int)(word & 0xff) : FA_OK;
}

}  // extern "C"
