// cuTensorMapEncodeTiled through the runtime's driver entry point, so the
// library does not link libcuda directly.
#include <cudaTypedefs.h>

#include <mutex>

#include "tensor_map.h"

namespace moda {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_once;

void resolve() {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
}

}  // namespace

static CUresult encode_bf16(CUtensorMap* m, const void* base, int rank, const uint64_t* dims,
                            const uint64_t* strides_bytes, const uint32_t* box,
                            CUtensorMapSwizzle swizzle,
                            CUtensorMapL2promotion promotion = CU_TENSOR_MAP_L2_PROMOTION_L2_256B) {
  std::call_once(g_once, resolve);
  if (!g_encode) return CUDA_ERROR_NOT_FOUND;
  cuuint64_t gdim[5];
  cuuint64_t gstride[4];
  cuuint32_t bdim[5], estride[5];
  for (int i = 0; i < rank; ++i) {
    gdim[i] = dims[i];
    bdim[i] = box[i];
    estride[i] = 1;
  }
  for (int i = 0; i + 1 < rank; ++i) gstride[i] = strides_bytes[i];
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void*>(base),
                  gdim, gstride, bdim, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                  promotion, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

CUresult encode_bf16_sw128(CUtensorMap* m, const void* base, int rank, const uint64_t* dims,
                           const uint64_t* strides_bytes, const uint32_t* box,
                           int l2_promotion_bytes) {
  return encode_bf16(m, base, rank, dims, strides_bytes, box, CU_TENSOR_MAP_SWIZZLE_128B,
                     l2_promotion_bytes == 128 ? CU_TENSOR_MAP_L2_PROMOTION_L2_128B
                                               : CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
}

CUresult encode_bf16_plain(CUtensorMap* m, const void* base, int rank, const uint64_t* dims,
                           const uint64_t* strides_bytes, const uint32_t* box) {
  return encode_bf16(m, base, rank, dims, strides_bytes, box, CU_TENSOR_MAP_SWIZZLE_NONE);
}

}  // namespace moda
