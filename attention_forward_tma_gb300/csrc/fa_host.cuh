// fa_host.cuh -- host helpers shared by the translation units of the library:
// the driver's tensor-map encoder, 3-D tensor maps over [tokens, heads, d]
// tensors, head-count checks and pointer alignment.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "fa.h"
#include "fa_fwd.cuh"

namespace fa_host {

// ------------------------------------------------------------------ driver entry point
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_fn() {
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

// 3-D map over a [tokens, heads, d] tensor of 16-bit elements: x = d (contiguous),
// y = head, z = token. Box = 64 x box_heads x (128 / box_heads): one 128-byte
// slab of a 128-row tile whose row r is token r / box_heads, head r % box_heads
// (box_heads = G packs the query heads of one K/V group; K and V use 1).
// 128-byte swizzle; rows outside the tensor read as 0.
inline int make_map(CUtensorMap* m, const void* base, long long tokens, int heads, int d, int box_heads, bool f16) {
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

// 3-D map over an fp32 [tokens, heads, d] tensor for tiled reduce-adds: box =
// 32 x box_heads x (128 / box_heads) (one 128-byte column slab of a packed
// 128-row tile), 128-byte swizzle.
inline int make_map_f32(CUtensorMap* m, void* base, long long tokens, int heads, int d, int box_heads) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return FA_ERR_CUDA;
  const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)heads, (cuuint64_t)tokens};
  const cuuint64_t strides[2] = {(cuuint64_t)d * 4, (cuuint64_t)heads * d * 4};
  const cuuint32_t box[3] = {32, (cuuint32_t)box_heads, (cuuint32_t)(fa::kBlockM / box_heads)};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

// H_kv must divide H, and the group size G = H / H_kv must divide the 128 rows of
// a Q tile (a power of two up to 128). Sets gshift = log2(G).
inline int check_heads(int H, int Hkv, int* gshift) {
  if (H <= 0 || Hkv <= 0 || H % Hkv != 0) return FA_ERR_INVALID_ARG;
  const int G = H / Hkv;
  if (G > fa::kBlockM || (G & (G - 1)) != 0) return FA_ERR_UNSUPPORTED;
  int sh = 0;
  while ((1 << sh) < G) ++sh;
  *gshift = sh;
  return FA_OK;
}

inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// The device status word of the backward translation unit (each translation unit
// has its own copy of the status variable): returns it and clears it.
int bwd_take_status(unsigned long long* word);

// The clock-stamp buffer set by fa_trace_configure (tracing builds; else null, 0).
void trace_target(unsigned long long** buf, int* ctas);
// Process-wide options of fa_set_option read by the backward translation unit.
bool bwd_deterministic();
int bwd_section_override();   // > 0: pairs per L2 section of the backward grid (tests, tuning)
int persistent_mode();        // FA_OPT_PERSISTENT (-1 = the default)
// Stream-ordered allocation from the library's own pool on the current device (memory
// kept between calls); free with cudaFreeAsync.
cudaError_t alloc_async(void** ptr, size_t bytes, cudaStream_t s);
// Trim the pools of alloc_async to what pending allocations still need.
cudaError_t release_pools();
unsigned long long wait_timeout_ns();

}  // namespace fa_host
