// Host-side TMA tensor-map encoding through the driver entry point (no link
// against libcuda; the runtime hands out the driver symbol).
#include <cudaTypedefs.h>

#include <mutex>

#include "tc_ptx.cuh"

namespace ulysses {

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

int make_tmap_bf16_3d(CUtensorMap* map, const void* base, int64_t S, int heads, int D, int rows) {
  auto fn = encode_fn();
  if (!fn) return set_error(ULYSSES_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
  if ((reinterpret_cast<uintptr_t>(base) & 15u) != 0)
    return set_error(ULYSSES_ERR_INVALID, "TMA base must be 16-byte aligned");
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)S, (cuuint64_t)heads};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)S * D * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return set_error(ULYSSES_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return ULYSSES_OK;
}

static int encode(CUtensorMap* map, CUtensorMapDataType dt, const void* base, const cuuint64_t* dims,
                  const cuuint64_t* strides, const cuuint32_t* box, CUtensorMapSwizzle sw) {
  auto fn = encode_fn();
  if (!fn) return set_error(ULYSSES_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
  if ((reinterpret_cast<uintptr_t>(base) & 15u) != 0)
    return set_error(ULYSSES_ERR_INVALID, "TMA base must be 16-byte aligned");
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, dt, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return set_error(ULYSSES_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return ULYSSES_OK;
}

int make_tmap_bf16_seq(CUtensorMap* map, const void* base, int64_t S, int heads, int row_heads, int D, int rows) {
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)heads, (cuuint64_t)S};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)row_heads * D * 2};
  cuuint32_t box[3] = {64, 1, (cuuint32_t)rows};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

int make_tmap_f32_seq(CUtensorMap* map, const void* base, int64_t S, int heads, int row_heads, int D, int rows) {
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)heads, (cuuint64_t)S};
  cuuint64_t strides[2] = {(cuuint64_t)D * 4, (cuuint64_t)row_heads * D * 4};
  cuuint32_t box[3] = {(cuuint32_t)D, 1, (cuuint32_t)rows};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
}

}  // namespace ulysses
