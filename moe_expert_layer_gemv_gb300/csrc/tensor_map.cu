// tensor_map.cu -- host-side encoding of the tiled tensor maps the GEMV stages
// load their int4 weight boxes through (cp.async.bulk.tensor), by the driver's
// cuTensorMapEncodeTiled, looked up once through the runtime's entry-point
// query (no link against the driver library).
#include <cudaTypedefs.h>

#include "launch.h"

namespace moe {

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_entry() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

}  // namespace

bool encode_map(CUtensorMap* m, CUtensorMapDataType type, int rank, const void* base,
                const uint64_t* dims, const uint64_t* strides, const uint32_t* box,
                CUtensorMapSwizzle swizzle) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_entry();
  if (fn == nullptr || rank < 2 || rank > 3) return false;
  cuuint64_t gd[3], gs[2];
  cuuint32_t bx[3], estr[3] = {1, 1, 1};
  for (int i = 0; i < rank; ++i) {
    gd[i] = dims[i];
    bx[i] = box[i];
    if (i + 1 < rank) gs[i] = strides[i];
  }
  return fn(m, type, (cuuint32_t)rank, const_cast<void*>(base), gd, gs, bx, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_map_2d(CUtensorMap* m, CUtensorMapDataType type, int elem_bytes, const void* base,
                   uint64_t rows, uint64_t cols, uint32_t box_cols, uint32_t box_rows,
                   CUtensorMapSwizzle swizzle) {
  const uint64_t dims[2] = {cols, rows};
  const uint64_t strides[1] = {cols * (uint64_t)elem_bytes};
  const uint32_t box[2] = {box_cols, box_rows};
  return encode_map(m, type, 2, base, dims, strides, box, swizzle);
}

}  // namespace moe
