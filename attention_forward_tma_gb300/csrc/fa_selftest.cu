// fa_selftest.cu -- diagnostic kernels behind include/fa_selftest.h. They reuse
// the attention kernel's own building blocks (TMA maps, descriptors, MMA issue
// helpers, exponentials, bounded waits) on single pieces of work.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstring>

#include "fa.h"
#include "fa_fwd.cuh"
#include "fa_selftest.h"

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

int tile_map(CUtensorMap* m, const void* base, int rows, int d, bool f16) {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return FA_ERR_CUDA;
  const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)rows, 1};
  const cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)d * 2 * rows};
  const cuuint32_t box[3] = {64, 128, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = reinterpret_cast<EncodeTiledFn>(fn)(
      m, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
      strides, box, estr,
      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

struct TileMaps {
  CUtensorMap q, k, v;
};

template <int D, bool F16>
__global__ void __launch_bounds__(128, 1) mma_tile_kernel(const __grid_constant__ TileMaps maps,
                                                           const uint32_t* __restrict__ p_pairs,
                                                           float* __restrict__ s_out, float* __restrict__ o_out,
                                                           unsigned long long timeout_ns) {
  using namespace fa;
  using L = Layout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sQ = smem_u32(smem), sK = sQ + L::kTileBytes, sV = sK + L::kTileBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + 3 * L::kTileBytes);
  uint32_t* slot = reinterpret_cast<uint32_t*>(smem + 3 * L::kTileBytes + 64);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + 3 * L::kTileBytes + 68);
  const uint32_t bLoad = smem_u32(&bars[0]), bMma = smem_u32(&bars[1]);
  const int tid = threadIdx.x, warp = tid >> 5;
  if (tid == 0) {
    *abort_flag = 0;
    mbar_init(bLoad, 1);
    mbar_init(bMma, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *slot;
  const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
  Waiter w{abort_flag, timeout_ns, 7};
  bool ok = true;
  if (warp == 0) {  // whole warp waits; one elected lane issues
    const bool leader = elect_one();
    if (leader) {
      mbar_arrive_expect_tx(bLoad, 3 * L::kTileBytes);
      for (int c = 0; c < L::kHalves; ++c) {
        tma_load_3d(sQ + c * L::kSlabBytes, &maps.q, c * 64, 0, 0, bLoad);
        tma_load_3d(sK + c * L::kSlabBytes, &maps.k, c * 64, 0, 0, bLoad);
        tma_load_3d(sV + c * L::kSlabBytes, &maps.v, c * 64, 0, 0, bLoad);
      }
    }
    __syncwarp();
    ok = w.wait(bLoad, 0, 0, 0);
    if (leader) {
      if (ok) {
        tc_fence_after();
        issue_qk<D, F16>(tmem + L::col_s(0), smem_desc_sw128(sQ, 16, 1024), smem_desc_sw128(sK, 16, 1024));
      }
      mma_commit(bMma);
    }
    __syncwarp();
  }
  ok = w.wait(bMma, 0, 1, 0) && !*abort_flag;
  tc_fence_after();
  const int r = tid;
  if (ok) {
    uint32_t u[128];
    for (int c = 0; c < 4; ++c) tmem_ld32(tmem + lane_base + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&u[c * 32]));
    tmem_wait_ld();
    for (int c = 0; c < 128; ++c) s_out[r * 128 + c] = __uint_as_float(u[c]);
    uint32_t pk[64];
    for (int c = 0; c < 64; ++c) pk[c] = p_pairs[r * 64 + c];
    tmem_st32(tmem + lane_base + 64, *reinterpret_cast<const uint32_t(*)[32]>(&pk[0]));
    tmem_st32(tmem + lane_base + 96, *reinterpret_cast<const uint32_t(*)[32]>(&pk[32]));
    tmem_wait_st();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) {
    if (elect_one()) {
      if (ok) issue_pv<D, 0, kBlockN, F16>(tmem + L::col_o(0), tmem + L::col_s(0) + 64,
                                           smem_desc_sw128(sV, L::kSlabBytes, 1024), false);
      mma_commit(bMma);
    }
    __syncwarp();
  }
  ok = w.wait(bMma, 1, 1, 1) && ok;
  tc_fence_after();
  if (ok) {
    for (int c = 0; c < D / 32; ++c) {
      uint32_t u[32];
      tmem_ld32(tmem + lane_base + L::col_o(0) + c * 32, u);
      tmem_wait_ld();
      for (int e = 0; e < 32; ++e) o_out[r * D + c * 32 + e] = __uint_as_float(u[e]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

__global__ void exp2_kernel(const float* x, float* y, int n, int use_poly) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) {
    if (use_poly == 2) {  // the packed pair form used inside the softmax
      float lo, hi;
      fa::unpack2(fa::exp2_poly2(fa::pack2(x[i], x[i])), lo, hi);
      y[i] = lo;
    } else {
      y[i] = use_poly ? fa::exp2_poly(x[i]) : fa::ex2_approx(x[i]);
    }
  }
}

__global__ void wait_timeout_kernel(unsigned long long timeout_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    fa::mbar_init(fa::smem_u32(&bar), 1);  // nothing ever arrives on it
    fa::fence_mbar_init();
  }
  __syncthreads();
  fa::Waiter w{&abort_flag, timeout_ns, 7};  // all 32 lanes wait together
  w.wait(fa::smem_u32(&bar), 0, 99, -1);
}

int read_and_clear_status() {
  unsigned long long word = 0;
  if (cudaMemcpyFromSymbol(&word, fa::g_fa_status, sizeof word) != cudaSuccess) return FA_ERR_CUDA;
  if (word) {
    const unsigned long long zero = 0;
    if (cudaMemcpyToSymbol(fa::g_fa_status, &zero, sizeof zero) != cudaSuccess) return FA_ERR_CUDA;
  }
  return (int)(word & 0xff);
}

template <int D, bool F16>
void launch_mma_tile(const TileMaps& maps, const void* p, float* s_out, float* o_out, cudaStream_t s) {
  const int smem = 3 * fa::Layout<D>::kTileBytes + 128 + 1024;
  cudaFuncSetAttribute(mma_tile_kernel<D, F16>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  mma_tile_kernel<D, F16><<<1, 128, smem, s>>>(maps, static_cast<const uint32_t*>(p), s_out, o_out, 2000000000ull);
}

bool is_sm103() {
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  return major == 10 && minor == 3;
}

}  // namespace

extern "C" {

int fa_selftest_mma_tile(const void* q, const void* k, const void* v, const void* p, float* s_out, float* o_out,
                         int d, int dtype, void* stream) {
  if (!q || !k || !v || !p || !s_out || !o_out) return FA_ERR_INVALID_ARG;
  if (dtype != FA_DTYPE_BF16 && dtype != FA_DTYPE_FP16) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if (!is_sm103()) return FA_ERR_UNSUPPORTED;
  const bool f16 = dtype == FA_DTYPE_FP16;
  TileMaps maps;
  std::memset(&maps, 0, sizeof maps);
  int st;
  if ((st = tile_map(&maps.q, q, 128, d, f16)) != FA_OK || (st = tile_map(&maps.k, k, 128, d, f16)) != FA_OK ||
      (st = tile_map(&maps.v, v, 128, d, f16)) != FA_OK)
    return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (d == 128) {
    if (f16) launch_mma_tile<128, true>(maps, p, s_out, o_out, s);
    else launch_mma_tile<128, false>(maps, p, s_out, o_out, s);
  } else {
    if (f16) launch_mma_tile<64, true>(maps, p, s_out, o_out, s);
    else launch_mma_tile<64, false>(maps, p, s_out, o_out, s);
  }
  if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return FA_ERR_CUDA;
  return read_and_clear_status();
}

int fa_selftest_exp2(const float* x, float* y, int n, int use_poly, void* stream) {
  if (!x || !y || n < 0) return FA_ERR_INVALID_ARG;
  if (n == 0) return FA_OK;
  exp2_kernel<<<(n + 255) / 256, 256, 0, static_cast<cudaStream_t>(stream)>>>(x, y, n, use_poly);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int fa_selftest_wait_timeout(unsigned long long timeout_ns, void* stream) {
  if (timeout_ns < 1000ull || timeout_ns > 10000000000ull) return FA_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  wait_timeout_kernel<<<1, 32, 0, s>>>(timeout_ns);
  if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return FA_ERR_CUDA;
  return read_and_clear_status();
}

}  // extern "C"
