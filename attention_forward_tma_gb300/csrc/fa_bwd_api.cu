// fa_bwd_api.cu -- host side of fa_bwd (include/fa.h): argument checks, the
// temporary buffer (fp32 dQ accumulator, packed D and base-2 LSE), tensor maps and
// the three launches: preprocessing, the backward kernel, the dQ conversion.
#include <cuda.h>
#include <cuda_runtime.h>

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
int launch(const fa::BwdParams& p, cudaStream_t s) {
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
  kern<<<p.num_tasks, fa::kBwdThreads, L::kAlloc, s>>>(p);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

template <int D, bool F>
int launch_c(const fa::BwdParams& p, bool causal, cudaStream_t s) {
  return causal ? launch<D, true, F>(p, s) : launch<D, false, F>(p, s);
}

template <int D, bool F>
int pre_post(bool post, const void* o, const void* dout, const float* lse, float* lse2, float* dsum,
             float* dq_acc, void* dq, int B, int H, int gshift, int Nq, int mpad, cudaStream_t s) {
  if (!post) {
    const long long rows = (long long)B * Nq * H;
    fa::fa_bwd_pre_kernel<D, F><<<(unsigned)((rows + 7) / 8), 256, 0, s>>>(
        static_cast<const uint16_t*>(o), static_cast<const uint16_t*>(dout), lse, lse2, dsum, dq_acc, B, H, gshift,
        Nq, mpad);
  } else {
    const long long n4 = (long long)B * Nq * H * D / 4;
    fa::fa_bwd_post_kernel<F><<<(unsigned)((n4 + 255) / 256), 256, 0, s>>>(
        reinterpret_cast<const float4*>(dq_acc), static_cast<uint2*>(dq), n4);
  }
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int pre_post_any(bool post, int d, bool f16, const void* o, const void* dout, const float* lse, float* lse2,
                 float* dsum, float* dq_acc, void* dq, int B, int H, int gshift, int Nq, int mpad,
                 cudaStream_t s) {
  if (d == 128)
    return f16 ? pre_post<128, true>(post, o, dout, lse, lse2, dsum, dq_acc, dq, B, H, gshift, Nq, mpad, s)
               : pre_post<128, false>(post, o, dout, lse, lse2, dsum, dq_acc, dq, B, H, gshift, Nq, mpad, s);
  return f16 ? pre_post<64, true>(post, o, dout, lse, lse2, dsum, dq_acc, dq, B, H, gshift, Nq, mpad, s)
             : pre_post<64, false>(post, o, dout, lse, lse2, dsum, dq_acc, dq, B, H, gshift, Nq, mpad, s);
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
  int dev = 0, n = 0, major = 0, minor = 0;
  if (cudaGetDeviceCount(&n) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    return FA_ERR_NO_DEVICE;
  }
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return FA_ERR_CUDA;
  if (major != 10 || minor != 3) return FA_ERR_UNSUPPORTED;
  const bool f16 = dtype == FA_DTYPE_FP16;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  fa::BwdParams p;
  std::memset(&p, 0, sizeof p);
  const int G = H / H_kv;
  if ((st = make_map(&p.tm_q, q, tokens, H, d, G, f16)) != FA_OK ||
      (st = make_map(&p.tm_do, dout, tokens, H, d, G, f16)) != FA_OK ||
      (st = make_map(&p.tm_k, k, tokens_k, H_kv, d, 1, f16)) != FA_OK ||
      (st = make_map(&p.tm_v, v, tokens_k, H_kv, d, 1, f16)) != FA_OK)
    return st;

  // temporary buffer: dQ accumulator (fp32 [tokens, H, d], zeroed by the
  // preprocessing kernel), then packed base-2 LSE and D ([B, H_kv, mpad] each,
  // zeroed here so padding rows read 0)
  const size_t acc_bytes = (size_t)tokens * H * d * sizeof(float);
  const size_t vec_bytes = ((size_t)B * H_kv * mpad * sizeof(float) + 255) / 256 * 256;
  const bool det = fa_host::bwd_deterministic();
  const int ntiles = (int)(mpad / 128);
  const size_t sem_bytes = det ? ((size_t)B * H_kv * ntiles * sizeof(int) + 255) / 256 * 256 : 0;
  void* ws = nullptr;
  if (cudaMallocAsync(&ws, acc_bytes + 2 * vec_bytes + sem_bytes, s) != cudaSuccess) {
    cudaGetLastError();
    return FA_ERR_CUDA;
  }
  float* dq_acc = static_cast<float*>(ws);
  float* lse2 = reinterpret_cast<float*>(static_cast<char*>(ws) + acc_bytes);
  float* dsum = reinterpret_cast<float*>(static_cast<char*>(ws) + acc_bytes + vec_bytes);
  int* sem = det ? reinterpret_cast<int*>(static_cast<char*>(ws) + acc_bytes + 2 * vec_bytes) : nullptr;
  if (cudaMemsetAsync(lse2, 0, 2 * vec_bytes + sem_bytes, s) != cudaSuccess) st = FA_ERR_CUDA;
  if (st == FA_OK)
    st = pre_post_any(false, d, f16, o, dout, lse, lse2, dsum, dq_acc, nullptr, B, H, gshift, N_q, (int)mpad, s);
  if (st == FA_OK) st = fa_host::make_map_f32(&p.tm_dq, dq_acc, tokens, H, d, G);
  if (st == FA_OK) {
    p.lse2 = lse2;
    p.dsum = dsum;
    p.dq_acc = dq_acc;
    p.dk = static_cast<uint16_t*>(dk);
    p.dv = static_cast<uint16_t*>(dv);
    p.B = B; p.H = H; p.Hkv = H_kv; p.gshift = gshift; p.Nq = N_q; p.Nk = N_kv;
    p.nkb = (int)nkb;
    p.mpad = (int)mpad;
    p.num_tasks = (int)(B * H_kv * nkb);
    p.scale = scale;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.timeout_ns = fa_host::wait_timeout_ns();
    p.sem = sem;
    p.ntiles = ntiles;
    fa_host::trace_target(&p.trace, &p.trace_ctas);
    if (d == 128)
      st = f16 ? launch_c<128, true>(p, causal != 0, s) : launch_c<128, false>(p, causal != 0, s);
    else
      st = f16 ? launch_c<64, true>(p, causal != 0, s) : launch_c<64, false>(p, causal != 0, s);
  }
  if (st == FA_OK)
    st = pre_post_any(true, d, f16, nullptr, nullptr, nullptr, nullptr, nullptr, dq_acc, dq, B, H, gshift, N_q,
                      (int)mpad, s);
  if (cudaFreeAsync(ws, s) != cudaSuccess && st == FA_OK) st = FA_ERR_CUDA;
  return st;
}

}  // extern "C"
