// fa_api.cu -- host side of the C ABI declared in include/fa.h: argument checks,
// TMA tensor maps, the varlen longest-first schedule kernel, kernel launches and
// the device status word.
#include <cuda.h>
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "fa.h"
#include "fa_fwd.cuh"
#include "fa_selftest.h"

namespace {

// ------------------------------------------------------------------ options
struct Options {
  float tau = 8.0f;
  unsigned long long timeout_ns = 2000000000ull;
  int persistent = -1;   // -1: default (work stealing)
  int emu_groups = 0;
};
Options g_opt;

// tracing builds: where fa_fwd / fa_fwd_varlen write their clock stamps
unsigned long long* g_trace_buf = nullptr;
int g_trace_ctas = 0;

// ------------------------------------------------------------------ driver entry point
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// ------------------------------------------------------------------ per-device facts
struct DevInfo {
  bool init = false;
  bool supported = false;
  int sm_count = 0;
  long long l2_bytes = 0;
  bool attr_done[2][2][2][2] = {};   // [d == 128][causal][emulation][fp16]
  int attr_status[2][2][2][2] = {};
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

// 3-D map over a [tokens, heads, d] tensor of 16-bit elements: x = d (contiguous),
// y = head, z = token. Box = 64 x box_heads x (128 / box_heads): one 128-byte
// slab of a 128-row tile whose row r is token r / box_heads, head r % box_heads
// (box_heads = G packs the query heads of one K/V group; K and V use 1).
// 128-byte swizzle; rows outside the tensor read as 0.
int make_map(CUtensorMap* m, const void* base, long long tokens, int heads, int d, int box_heads, bool f16) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return FA_ERR_CUDA;
  const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)heads, (cuuint64_t)tokens};
  const cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)heads * d * 2};
  const cuuint32_t box[3] = {64, (cuuint32_t)box_heads, (cuuint32_t)(fa::kBlockM / box_heads)};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                   const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

// The four maps of one call: Q and O with H heads in boxes of G, K and V with H_kv heads.
int make_maps(fa::FwdParams& p, const void* q, const void* k, const void* v, void* o, long long tokens, int H,
              int Hkv, int d, bool f16) {
  const int G = H / Hkv;
  int st;
  if ((st = make_map(&p.tm_q, q, tokens, H, d, G, f16)) != FA_OK ||
      (st = make_map(&p.tm_k, k, tokens, Hkv, d, 1, f16)) != FA_OK ||
      (st = make_map(&p.tm_v, v, tokens, Hkv, d, 1, f16)) != FA_OK ||
      (st = make_map(&p.tm_o, o, tokens, H, d, G, f16)) != FA_OK)
    return st;
  return FA_OK;
}

// H_kv must divide H, and the group size G = H / H_kv must divide the 128 rows of
// a Q tile (a power of two up to 128). Sets gshift = log2(G).
int check_heads(int H, int Hkv, int* gshift) {
  if (H <= 0 || Hkv <= 0 || H % Hkv != 0) return FA_ERR_INVALID_ARG;
  const int G = H / Hkv;
  if (G > fa::kBlockM || (G & (G - 1)) != 0) return FA_ERR_UNSUPPORTED;
  int sh = 0;
  while ((1 << sh) < G) ++sh;
  *gshift = sh;
  return FA_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

template <int D, bool C, bool E, bool F>
int launch_fwd(DevInfo* dev, const fa::FwdParams& p, int grid, cudaStream_t stream) {
  using L = fa::Layout<D>;
  auto kern = fa::fa_fwd_kernel<D, C, E, F>;
  const int di = D == 128 ? 1 : 0, ci = C ? 1 : 0, ei = E ? 1 : 0, fi = F ? 1 : 0;
  {
    std::lock_guard<std::mutex> lk(g_dev_mu);
    if (!dev->attr_done[di][ci][ei][fi]) {
      int st = FA_OK;
      cudaFuncAttributes fa_attr;
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmemAlloc) != cudaSuccess ||
          cudaFuncGetAttributes(&fa_attr, kern) != cudaSuccess)
        st = FA_ERR_CUDA;
      // the warpgroup register split (192/192/48/80) needs exactly 128 registers
      // per thread at launch
      else if (fa_attr.numRegs != 128)
        st = FA_ERR_UNSUPPORTED;
      dev->attr_status[di][ci][ei][fi] = st;
      dev->attr_done[di][ci][ei][fi] = true;
    }
    if (dev->attr_status[di][ci][ei][fi] != FA_OK) return dev->attr_status[di][ci][ei][fi];
  }
  kern<<<grid, fa::kThreads, L::kSmemAlloc, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

template <int D, bool C, bool F>
int dispatch_emu(DevInfo* dev, const fa::FwdParams& p, int grid, cudaStream_t s) {
  return p.emu_groups > 0 ? launch_fwd<D, C, true, F>(dev, p, grid, s) : launch_fwd<D, C, false, F>(dev, p, grid, s);
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

// One CTA: enumerate the (sequence, 256-row block) work tiles, bucket them by
// their number of K/V blocks, and write them longest first, each followed by
// all Hkv K/V heads ("FlashAttention-4（下）" (argus lesson 7), section "6. LPT 调度":
// sort work tiles by their cost, write a virtual -> actual map). Rows are packed
// (sequence position, query head of the group): a sequence of length L has
// L << gshift rows, and row r of a block sits at position r >> gshift.
__global__ void __launch_bounds__(1024) fa_varlen_schedule_kernel(const int* cu, int num_seqs, int Hkv, int gshift,
                                                                  int causal, int capacity, int4* tasks, int* count) {
  __shared__ int hist[kSchedBuckets];
  __shared__ int total_pairs;
  for (int i = threadIdx.x; i < kSchedBuckets; i += blockDim.x) hist[i] = 0;
  if (threadIdx.x == 0) total_pairs = 0;
  __syncthreads();
  auto cost_of = [&](int L, int m) {
    const int kmax = causal ? min(((m * kTaskRows + kTaskRows - 1) >> gshift) + 1, L) : L;
    return min((kmax + kBlockN - 1) / kBlockN, kSchedBuckets - 1);
  };
  for (int s = threadIdx.x; s < num_seqs; s += blockDim.x) {
    const int L = max(cu[s + 1] - cu[s], 0);
    const int nm = ((L << gshift) + kTaskRows - 1) / kTaskRows;
    for (int m = 0; m < nm; ++m) atomicAdd(&hist[cost_of(L, m)], 1);
    atomicAdd(&total_pairs, nm);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // exclusive scan from the most expensive bucket down: hist[c] becomes the
    // first slot of bucket c
    int run = 0;
    for (int c = kSchedBuckets - 1; c >= 0; --c) {
      const int n = hist[c];
      hist[c] = run;
      run += n;
    }
    const long long n_tasks = (long long)total_pairs * Hkv;
    *count = (int)(n_tasks < capacity ? n_tasks : capacity);
  }
  __syncthreads();
  for (int s = threadIdx.x; s < num_seqs; s += blockDim.x) {
    const int L = max(cu[s + 1] - cu[s], 0);
    const int nm = ((L << gshift) + kTaskRows - 1) / kTaskRows;
    for (int m = 0; m < nm; ++m) {
      const int c = cost_of(L, m);
      const int slot = atomicAdd(&hist[c], 1);
      for (int h = 0; h < Hkv; ++h) {
        const long long ti = (long long)slot * Hkv + h;
        if (ti < capacity) tasks[ti] = make_int4(s, h, m, c);
      }
    }
  }
}
}  // namespace fa

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

// ------------------------------------------------------------------ C ABI
extern "C" {

int fa_version(void) { return 100; }

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
    default:
      return FA_ERR_INVALID_ARG;
  }
}

int fa_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int H_kv, int N,
               int d, float scale, int causal, int dtype, void* stream) {
  if (!q || !k || !v || !o) return FA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || (lse && !aligned(lse, 4)))
    return FA_ERR_INVALID_ARG;
  if (B <= 0 || H <= 0 || H_kv <= 0 || N <= 0) return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  if (dtype != FA_DTYPE_BF16 && dtype != FA_DTYPE_FP16) return FA_ERR_INVALID_ARG;
  int gshift = 0;
  int st = check_heads(H, H_kv, &gshift);
  if (st != FA_OK) return st;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  const long long tokens = (long long)B * N;
  if (tokens * H > INT_MAX) return FA_ERR_INVALID_ARG;  // 32-bit row and LSE indexing
  DevInfo* dev = nullptr;
  if ((st = device_info(&dev)) != FA_OK) return st;
  const bool f16 = dtype == FA_DTYPE_FP16;

  fa::FwdParams p;
  std::memset(&p, 0, sizeof p);
  if ((st = make_maps(p, q, k, v, o, tokens, H, H_kv, d, f16)) != FA_OK) return st;
  p.o = static_cast<uint16_t*>(o);
  p.lse = lse;
  p.B = B; p.H = H; p.N = N;
  p.Hkv = H_kv;
  p.gshift = gshift;
  p.total_tokens = (int)tokens;
  // tasks of 256 packed rows; a (b, kv head) has N * G rows
  p.num_m = (int)((((long long)N << gshift) + fa::kTaskRows - 1) / fa::kTaskRows);
  const long long ntask = (long long)B * H_kv * p.num_m;
  if (ntask > INT_MAX) return FA_ERR_INVALID_ARG;
  p.num_tasks = (int)ntask;
  const long long kv_bytes = 4LL * N * d;                       // K + V of one (b, kv head)
  long long group = (dev->l2_bytes / 2) / (kv_bytes > 0 ? kv_bytes : 1);
  if (group < 1) group = 1;
  if (group > (long long)B * H_kv) group = (long long)B * H_kv;
  p.lpt_group = (int)group;
  p.varlen = 0;
  fill_common(p, scale, f16);
  const int grid = grid_for(p, dev, p.num_tasks);
  return dispatch(dev, p, d, causal != 0, f16, grid, static_cast<cudaStream_t>(stream));
}

int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
           float scale, int causal, void* stream) {
  return fa_fwd_gqa(q, k, v, o, lse, B, H, H, N, d, scale, causal, FA_DTYPE_BF16, stream);
}

}  // extern "C"

namespace {
// Argument checks shared by the varlen entry points; *cap = the task-list
// capacity: H_kv * (ceil(T * G / 256) + num_seqs) tiles of 256 packed rows.
int varlen_check(const void* q, const void* k, const void* v, void* o, float* lse, const int* cu_seqlens,
                 int num_seqs, int total_tokens, int max_seqlen, int H, int H_kv, int d, float scale, int causal,
                 int dtype, int* gshift, long long* cap) {
  if (!q || !k || !v || !o || !cu_seqlens) return FA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || (lse && !aligned(lse, 4)) ||
      !aligned(cu_seqlens, 4))
    return FA_ERR_INVALID_ARG;
  if (num_seqs <= 0 || total_tokens <= 0 || max_seqlen <= 0 || H <= 0 || H_kv <= 0) return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  if (dtype != FA_DTYPE_BF16 && dtype != FA_DTYPE_FP16) return FA_ERR_INVALID_ARG;
  int st = check_heads(H, H_kv, gshift);
  if (st != FA_OK) return st;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if ((long long)total_tokens * H > INT_MAX) return FA_ERR_INVALID_ARG;
  *cap = (long long)H_kv *
         ((((long long)total_tokens << *gshift) + fa::kTaskRows - 1) / fa::kTaskRows + num_seqs);
  return FA_OK;
}

// Maps, schedule kernel and attention kernel of a varlen call whose task list
// lives in tasks[0, cap) with its count at *count.
int varlen_launch(DevInfo* dev, const void* q, const void* k, const void* v, void* o, float* lse,
                  const int* cu_seqlens, int num_seqs, int total_tokens, int H, int H_kv, int gshift, int d,
                  float scale, int causal, bool f16, int4* tasks, int* count, int cap, cudaStream_t s) {
  fa::FwdParams p;
  std::memset(&p, 0, sizeof p);
  int st = make_maps(p, q, k, v, o, total_tokens, H, H_kv, d, f16);
  if (st != FA_OK) return st;
  fa::fa_varlen_schedule_kernel<<<1, 1024, 0, s>>>(cu_seqlens, num_seqs, H_kv, gshift, causal, cap, tasks, count);
  if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
  p.o = static_cast<uint16_t*>(o);
  p.lse = lse;
  p.cu_seqlens = cu_seqlens;
  p.tasks = tasks;
  p.task_count = count;
  p.H = H;
  p.Hkv = H_kv;
  p.gshift = gshift;
  p.total_tokens = total_tokens;
  p.num_tasks = cap;
  p.varlen = 1;
  fill_common(p, scale, f16);
  const int grid = grid_for(p, dev, cap);
  return dispatch(dev, p, d, causal != 0, f16, grid, s);
}
}  // namespace

extern "C" {

int fa_fwd_varlen_gqa(const void* q, const void* k, const void* v, void* o, float* lse, const int* cu_seqlens,
                      int num_seqs, int total_tokens, int max_seqlen, int H, int H_kv, int d, float scale,
                      int causal, int dtype, void* stream) {
  int gshift = 0;
  long long cap = 0;
  int st = varlen_check(q, k, v, o, lse, cu_seqlens, num_seqs, total_tokens, max_seqlen, H, H_kv, d, scale, causal,
                        dtype, &gshift, &cap);
  if (st != FA_OK) return st;
  if (cap > INT_MAX) return FA_ERR_INVALID_ARG;
  DevInfo* dev = nullptr;
  if ((st = device_info(&dev)) != FA_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  void* ws = nullptr;
  const size_t ws_bytes = (size_t)cap * sizeof(int4) + 16;
  if (cudaMallocAsync(&ws, ws_bytes, s) != cudaSuccess) {
    cudaGetLastError();
    return FA_ERR_CUDA;
  }
  int4* tasks = static_cast<int4*>(ws);
  int* count = reinterpret_cast<int*>(static_cast<char*>(ws) + (size_t)cap * sizeof(int4));
  st = varlen_launch(dev, q, k, v, o, lse, cu_seqlens, num_seqs, total_tokens, H, H_kv, gshift, d, scale, causal,
                     dtype == FA_DTYPE_FP16, tasks, count, (int)cap, s);
  if (cudaFreeAsync(ws, s) != cudaSuccess && st == FA_OK) st = FA_ERR_CUDA;
  return st;
}

int fa_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse, const int* cu_seqlens,
                  int num_seqs, int total_tokens, int max_seqlen, int H, int d, float scale, int causal,
                  void* stream) {
  return fa_fwd_varlen_gqa(q, k, v, o, lse, cu_seqlens, num_seqs, total_tokens, max_seqlen, H, H, d, scale, causal,
                           FA_DTYPE_BF16, stream);
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

int fa_varlen_schedule(const int* cu_seqlens, int num_seqs, int H_kv, int group, int causal, int capacity,
                       void* tasks, int* count, void* stream) {
  if (!cu_seqlens || !tasks || !count || num_seqs <= 0 || H_kv <= 0 || capacity < 0 || (causal != 0 && causal != 1))
    return FA_ERR_INVALID_ARG;
  if (!aligned(tasks, 16) || !aligned(count, 4) || !aligned(cu_seqlens, 4)) return FA_ERR_INVALID_ARG;
  int gshift = 0;
  if (group <= 0) return FA_ERR_INVALID_ARG;
  int st = check_heads(H_kv * group, H_kv, &gshift);
  if (st != FA_OK) return st;
  DevInfo* dev = nullptr;
  if ((st = device_info(&dev)) != FA_OK) return st;
  fa::fa_varlen_schedule_kernel<<<1, 1024, 0, static_cast<cudaStream_t>(stream)>>>(
      cu_seqlens, num_seqs, H_kv, gshift, causal, capacity, static_cast<int4*>(tasks), count);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int fa_fwd_varlen_noalloc(const void* q, const void* k, const void* v, void* o, float* lse, const int* cu_seqlens,
                          int num_seqs, int total_tokens, int max_seqlen, int H, int d, float scale, int causal,
                          void* stream) {
  int gshift = 0;
  long long cap = 0;
  int st = varlen_check(q, k, v, o, lse, cu_seqlens, num_seqs, total_tokens, max_seqlen, H, H, d, scale, causal,
                        FA_DTYPE_BF16, &gshift, &cap);
  if (st != FA_OK) return st;
  if (cap > kNoAllocMaxTasks) return FA_ERR_CAPACITY;
  DevInfo* dev = nullptr;
  if ((st = device_info(&dev)) != FA_OK) return st;
  int4* scratch = nullptr;
  if ((st = noalloc_scratch(&scratch)) != FA_OK) return st;
  int4* tasks = scratch;
  int* count = reinterpret_cast<int*>(scratch + kNoAllocMaxTasks);
  return varlen_launch(dev, q, k, v, o, lse, cu_seqlens, num_seqs, total_tokens, H, H, gshift, d, scale, causal,
                       false, tasks, count, (int)cap, static_cast<cudaStream_t>(stream));
}

int fa_last_device_status(void* stream, unsigned long long* detail) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return FA_ERR_CUDA;
  unsigned long long word = 0;
  if (cudaMemcpyFromSymbol(&word, fa::g_fa_status, sizeof word) != cudaSuccess) return FA_ERR_CUDA;
  if (detail) *detail = word;
  if (word != 0) {
    const unsigned long long zero = 0;
    if (cudaMemcpyToSymbol(fa::g_fa_status, &zero, sizeof zero) != cudaSuccess) return FA_ERR_CUDA;
    return (int)(word & 0xff);
  }
  return FA_OK;
}

}  // extern "C"
