// fa_bwd_api.cu -- host side of fa_bwd (include/fa.h): argument checks, the
// temporary buffer (fp32 dQ accumulator, packed D and base-2 LSE), tensor maps and
// the three launches: preprocessing, the backward kernel, the dQ conversion.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <cstring>
#include <mutex>

#include "fa.h"
#include "fa_bwd.cuh"
#include "fa_host.cuh"

namespace {
using fa_host::aligned;
using fa_host::check_heads;
using fa_host::make_map;

constexpr int kMaxDevices = 64;
std::mutex g_mu;
// per device and kernel instance: 0 = not checked, 1 = ready, else the status to return
int g_ready[kMaxDevices][2][2][2];

template <int D, bool C, bool F>
int launch(const fa::BwdParams& p, int grid, cudaStream_t s) {
  using L = fa::BwdLayout<D>;
  auto kern = fa::fa_bwd_kernel<D, C, F>;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    int& r = g_ready[dev][D == 128][C][F];
    if (r == 0) {
      cudaFuncAttributes a;
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc) != cudaSuccess ||
          cudaFuncGetAttributes(&a, kern) != cudaSuccess)
        r = FA_ERR_CUDA;
      // the warpgroup register split (136/136/120/120) needs exactly 128 registers per
      // thread at launch
      else if (a.numRegs != 128)
        r = FA_ERR_UNSUPPORTED;
      else
        r = 1;
    }
    if (r != 1) return r;
  }
  kern<<<grid, fa::kBwdThreads, L::kAlloc, s>>>(p);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

template <int D, bool F>
int launch_c(const fa::BwdParams& p, int grid, bool causal, cudaStream_t s) {
  return causal ? launch<D, true, F>(p, grid, s) : launch<D, false, F>(p, grid, s);
}

// Shape of one call: fixed length (cu_q == nullptr: B sequences of N_q / N_kv rows) or
// variable length (B sequences given by cu_q / cu_k; N_q, N_kv the longest ones).
struct Shape {
  int B, H, H_kv, N_q, N_kv, d, gshift;
  long long tokens_q, tokens_k;
  const int* cu_q;
  const int* cu_k;
};

template <int D, bool F>
int pre_post(bool post, const void* o, const void* dout, const float* lse, float* lse2, float* dsum,
             float* dq_acc, void* dq, const Shape& sh, int mpad, const int* cu_ok, cudaStream_t s) {
  const long long rows = sh.tokens_q * sh.H;
  if (rows == 0) return FA_OK;
  if (!post) {
    const long long rows_per_block = 8LL * (32 / (D / 8));
    fa::fa_bwd_pre_kernel<D, F><<<(unsigned)((rows + rows_per_block - 1) / rows_per_block), 256, 0, s>>>(
        static_cast<const uint16_t*>(o), static_cast<const uint16_t*>(dout), lse, lse2, dsum, dq_acc, sh.tokens_q,
        sh.cu_q, sh.B, sh.H, sh.gshift, sh.N_q, mpad, cu_ok);
  } else {
    const long long n4 = rows * D / 4;
    fa::fa_bwd_post_kernel<F><<<(unsigned)((n4 + 255) / 256), 256, 0, s>>>(
        reinterpret_cast<const float4*>(dq_acc), static_cast<uint2*>(dq), n4, cu_ok);
  }
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int pre_post_any(bool post, bool f16, const void* o, const void* dout, const float* lse, float* lse2, float* dsum,
                 float* dq_acc, void* dq, const Shape& sh, int mpad, const int* cu_ok, cudaStream_t s) {
  if (sh.d == 128)
    return f16 ? pre_post<128, true>(post, o, dout, lse, lse2, dsum, dq_acc, dq, sh, mpad, cu_ok, s)
               : pre_post<128, false>(post, o, dout, lse, lse2, dsum, dq_acc, dq, sh, mpad, cu_ok, s);
  return f16 ? pre_post<64, true>(post, o, dout, lse, lse2, dsum, dq_acc, dq, sh, mpad, cu_ok, s)
             : pre_post<64, false>(post, o, dout, lse, lse2, dsum, dq_acc, dq, sh, mpad, cu_ok, s);
}

int device_check() {
  int dev = 0, n = 0, major = 0, minor = 0;
  if (cudaGetDeviceCount(&n) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    return FA_ERR_NO_DEVICE;
  }
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return FA_ERR_CUDA;
  return major == 10 && minor == 3 ? FA_OK : FA_ERR_UNSUPPORTED;
}

// The three launches of one backward call (arguments already checked).
int bwd_run(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
            void* dq, void* dk, void* dv, const Shape& sh, float scale, int causal, bool f16, cudaStream_t s) {
  const int d = sh.d;
  fa::BwdParams p;
  std::memset(&p, 0, sizeof p);
  const int G = sh.H / sh.H_kv;
  int st;
  if ((st = make_map(&p.tm_q, q, sh.tokens_q, sh.H, d, G, f16)) != FA_OK ||
      (st = make_map(&p.tm_do, dout, sh.tokens_q, sh.H, d, G, f16)) != FA_OK ||
      (st = make_map(&p.tm_k, k, sh.tokens_k, sh.H_kv, d, 1, f16)) != FA_OK ||
      (st = make_map(&p.tm_v, v, sh.tokens_k, sh.H_kv, d, 1, f16)) != FA_OK)
    return st;
  const long long mpad = (((long long)sh.N_q << sh.gshift) + 127) / 128 * 128;
  const long long nkb = (sh.N_kv + 127) / 128;

  // temporary buffer: dQ accumulator (fp32 [tokens, H, d], zeroed by the
  // preprocessing kernel), then packed base-2 LSE and D ([B, H_kv, mpad] each,
  // zeroed here so padding rows read 0), then the deterministic mode's counters
  const size_t acc_bytes = ((size_t)sh.tokens_q * sh.H * d * sizeof(float) + 255) / 256 * 256;
  const size_t vec_bytes = ((size_t)sh.B * sh.H_kv * mpad * sizeof(float) + 255) / 256 * 256;
  const bool det = fa_host::bwd_deterministic();
  const int ntiles = (int)(mpad / 128);
  const size_t sem_bytes = (det ? ((size_t)sh.B * sh.H_kv * ntiles * sizeof(int) + 255) / 256 * 256 : 0) + 256;
  void* ws = nullptr;
  if (fa_host::alloc_async(&ws, acc_bytes + 2 * vec_bytes + sem_bytes, s) != cudaSuccess) {
    cudaGetLastError();
    return FA_ERR_CUDA;
  }
  float* dq_acc = static_cast<float*>(ws);
  float* lse2 = reinterpret_cast<float*>(static_cast<char*>(ws) + acc_bytes);
  float* dsum = reinterpret_cast<float*>(static_cast<char*>(ws) + acc_bytes + vec_bytes);
  int* sem = det ? reinterpret_cast<int*>(static_cast<char*>(ws) + acc_bytes + 2 * vec_bytes) : nullptr;
  int* counter = reinterpret_cast<int*>(static_cast<char*>(ws) + acc_bytes + 2 * vec_bytes + sem_bytes - 256);
  // variable length: the check kernel's verdict on the sequence offsets, next to the counter
  int* cu_ok = sh.cu_q != nullptr ? counter + 1 : nullptr;
  if (cudaMemsetAsync(lse2, 0, 2 * vec_bytes + sem_bytes, s) != cudaSuccess) st = FA_ERR_CUDA;
  if (st == FA_OK && cu_ok != nullptr) {
    fa::fa_bwd_check_cu_kernel<<<1, 1024, 0, s>>>(sh.cu_q, sh.cu_k, sh.B, (int)sh.tokens_q, (int)sh.tokens_k,
                                                  sh.N_q, sh.N_kv, cu_ok);
    if (cudaGetLastError() != cudaSuccess) st = FA_ERR_CUDA;
  }
  if (st == FA_OK) st = pre_post_any(false, f16, o, dout, lse, lse2, dsum, dq_acc, nullptr, sh, (int)mpad, cu_ok, s);
  if (st == FA_OK && sh.tokens_q > 0) st = fa_host::make_map_f32(&p.tm_dq, dq_acc, sh.tokens_q, sh.H, d, G);
  if (st == FA_OK && sh.tokens_q > 0 && sh.tokens_k > 0 && nkb > 0) {
    p.lse2 = lse2;
    p.dsum = dsum;
    p.dq_acc = dq_acc;
    p.dk = static_cast<uint16_t*>(dk);
    p.dv = static_cast<uint16_t*>(dv);
    p.cu_q = sh.cu_q;
    p.cu_k = sh.cu_k;
    p.B = sh.B; p.H = sh.H; p.Hkv = sh.H_kv; p.gshift = sh.gshift; p.Nq = sh.N_q; p.Nk = sh.N_kv;
    p.nkb = (int)nkb;
    // L2 sections of about 512 CTAs (3 to 4 waves of 152): measured on B4 H16 N4096,
    // B1 H32 N16384 and grouped B4 H32/8 N4096 against sections of 64 to 4096 CTAs.
    // The deterministic mode keeps one section: there the key blocks of a pair take
    // turns at every Q tile, and running all of them at once makes them wait longest.
    const int pairs = sh.B * sh.H_kv;
    p.section = det ? pairs : std::min(pairs, std::max(1, (int)((512 + nkb / 2) / nkb)));
    if (fa_host::bwd_section_override() > 0) p.section = std::min(pairs, fa_host::bwd_section_override());
    p.mpad = (int)mpad;
    p.num_tasks = (int)(sh.B * sh.H_kv * nkb);
    p.scale = scale;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.timeout_ns = fa_host::wait_timeout_ns();
    p.sem = sem;
    p.ntiles = ntiles;
    p.task_counter = counter;
    p.cu_ok = cu_ok;
    fa_host::trace_target(&p.trace, &p.trace_ctas);
    // persistent CTAs, one per SM, claiming tasks in order (FA_OPT_PERSISTENT = 0: one
    // CTA per task)
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
      st = FA_ERR_CUDA;
    const int grid = fa_host::persistent_mode() == 0 ? p.num_tasks : std::min(p.num_tasks, std::max(sms, 1));
    if (st != FA_OK)
      ;
    else if (d == 128)
      st = f16 ? launch_c<128, true>(p, grid, causal != 0, s) : launch_c<128, false>(p, grid, causal != 0, s);
    else
      st = f16 ? launch_c<64, true>(p, grid, causal != 0, s) : launch_c<64, false>(p, grid, causal != 0, s);
  }
  if (st == FA_OK)
    st = pre_post_any(true, f16, nullptr, nullptr, nullptr, nullptr, nullptr, dq_acc, dq, sh, (int)mpad, cu_ok, s);
  if (cudaFreeAsync(ws, s) != cudaSuccess && st == FA_OK) st = FA_ERR_CUDA;
  return st;
}
}  // namespace

namespace fa_host {
int bwd_take_status(unsigned long long* word) {
  *word = 0;
  if (cudaMemcpyFromSymbol(word, fa::g_fa_status, sizeof *word) != cudaSuccess) return FA_ERR_CUDA;
  if (*word != 0) {
    const unsigned long long zero = 0;
    if (cudaMemcpyToSymbol(fa::g_fa_status, &zero, sizeof zero) != cudaSuccess) return FA_ERR_CUDA;
  }
  return FA_OK;
}
}  // namespace fa_host

extern "C" {

int fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse, void* dq,
           void* dk, void* dv, int B, int H, int H_kv, int N_q, int N_kv, int d, float scale, int causal, int dtype,
           void* stream) {
  if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv) return FA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(dout, 16) ||
      !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16) || !aligned(lse, 4))
    return FA_ERR_INVALID_ARG;
  if (B <= 0 || H <= 0 || H_kv <= 0 || N_q <= 0 || N_kv <= 0) return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  if (dtype != FA_DTYPE_BF16 && dtype != FA_DTYPE_FP16) return FA_ERR_INVALID_ARG;
  int gshift = 0;
  int st = check_heads(H, H_kv, &gshift);
  if (st != FA_OK) return st;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  const long long tokens = (long long)B * N_q, tokens_k = (long long)B * N_kv;
  if (tokens * H > INT_MAX || tokens_k * H_kv > INT_MAX) return FA_ERR_INVALID_ARG;
  const long long mpad = (((long long)N_q << gshift) + 127) / 128 * 128;
  const long long nkb = (N_kv + 127) / 128;
  if ((long long)B * H_kv * mpad > INT_MAX || (long long)B * H_kv * nkb > INT_MAX) return FA_ERR_INVALID_ARG;
  if ((st = device_check()) != FA_OK) return st;
  const Shape sh{B, H, H_kv, N_q, N_kv, d, gshift, tokens, tokens_k, nullptr, nullptr};
  return bwd_run(q, k, v, o, dout, lse, dq, dk, dv, sh, scale, causal, dtype == FA_DTYPE_FP16,
                 static_cast<cudaStream_t>(stream));
}

int fa_bwd_varlen(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                  void* dq, void* dk, void* dv, const int* cu_seqlens_q, const int* cu_seqlens_kv, int num_seqs,
                  int total_q, int total_kv, int max_seqlen_q, int max_seqlen_kv, int H, int H_kv, int d,
                  float scale, int causal, int dtype, void* stream) {
  if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv || !cu_seqlens_q || !cu_seqlens_kv)
    return FA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(dout, 16) ||
      !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16) || !aligned(lse, 4) || !aligned(cu_seqlens_q, 4) ||
      !aligned(cu_seqlens_kv, 4))
    return FA_ERR_INVALID_ARG;
  if (num_seqs <= 0 || total_q <= 0 || total_kv <= 0 || max_seqlen_q <= 0 || max_seqlen_kv <= 0 || H <= 0 ||
      H_kv <= 0)
    return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  if (dtype != FA_DTYPE_BF16 && dtype != FA_DTYPE_FP16) return FA_ERR_INVALID_ARG;
  int gshift = 0;
  int st = check_heads(H, H_kv, &gshift);
  if (st != FA_OK) return st;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if ((long long)total_q * H > INT_MAX || (long long)total_kv * H_kv > INT_MAX) return FA_ERR_INVALID_ARG;
  const long long mpad = (((long long)max_seqlen_q << gshift) + 127) / 128 * 128;
  const long long nkb = ((long long)max_seqlen_kv + 127) / 128;
  if ((long long)num_seqs * H_kv * mpad > INT_MAX || (long long)num_seqs * H_kv * nkb > INT_MAX)
    return FA_ERR_INVALID_ARG;
  if ((st = device_check()) != FA_OK) return st;
  const Shape sh{num_seqs, H, H_kv, max_seqlen_q, max_seqlen_kv, d, gshift, total_q, total_kv, cu_seqlens_q,
                 cu_seqlens_kv};
  return bwd_run(q, k, v, o, dout, lse, dq, dk, dv, sh, scale, causal, dtype == FA_DTYPE_FP16,
                 static_cast<cudaStream_t>(stream));
}

}  // extern "C"
