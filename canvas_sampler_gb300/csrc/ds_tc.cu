// Host side of the tensor-core kernels: the driver's tensor-map encoder (resolved once), the SM
// count, and 2-D tensor maps over row-major arrays.
#include <cudaTypedefs.h>

#include <cstdlib>
#include <mutex>

#include "ds_internal.h"

namespace ds {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_once;
int g_sms = 0;

void resolve() {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  int dev = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&g_sms, cudaDevAttrMultiProcessorCount, dev);
  tc_prepare_logits();
  tc_prepare_selfcond();
  tc_prepare_vocab_pass();
}

bool encode(CUtensorMap* map, CUtensorMapDataType type, uint32_t esize, const void* base,
            uint64_t rows, uint64_t cols, uint32_t box_rows, uint32_t box_cols,
            CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * esize};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return g_encode(map, type, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool pdl_enabled() {
  static const bool on = [] {
    const char* e = getenv("DS_PDL");
    return !(e && e[0] == '0');
  }();
  return on;
}

bool tc_available() {
  std::call_once(g_once, resolve);
  return g_encode != nullptr;
}

int tc_num_sms() {
  std::call_once(g_once, resolve);
  return g_sms;
}

bool tc_make_map_bf16(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                      uint32_t box_rows, uint32_t box_cols) {
  return tc_available() &&
         encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, rows, cols, box_rows, box_cols);
}

bool tc_make_map_bf16_sw64(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                           uint32_t box_rows, uint32_t box_cols) {
  return tc_available() && encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, rows, cols,
                                  box_rows, box_cols, CU_TENSOR_MAP_SWIZZLE_64B);
}

bool tc_make_map_f32(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                     uint32_t box_rows, uint32_t box_cols) {
  return tc_available() &&
         encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, base, rows, cols, box_rows, box_cols);
}

}  // namespace ds
