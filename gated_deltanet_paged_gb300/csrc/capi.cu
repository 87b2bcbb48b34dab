// capi.cu -- host-side helpers of the C ABI: device check, tensor-map
// encoding, status strings.
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"

namespace gdn_host {

int check_device(int* sm_count) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return GDN_ERR_CUDA;
  }
  int major = 0, minor = 0, sms = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return GDN_ERR_CUDA;
  }
  if (major != 10 || minor != 3) return GDN_ERR_UNSUPPORTED;
  if (sm_count) *sm_count = sms;
  return GDN_OK;
}

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    cudaGetLastError();
  });
  return fn;
}

int encode_tokens_map(CUtensorMap* map, const void* base, int64_t T, int64_t H, int64_t D) {
  auto fn = encode_fn();
  if (!fn) return GDN_ERR_CUDA;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(T)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(D * 2), static_cast<cuuint64_t>(H * D * 2)};
  cuuint32_t box[3] = {64, 1, 64};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? GDN_OK : GDN_ERR_CUDA;
}

// [T, H, D] bf16 tokens with 32 x 1 x 32 boxes and the 64-byte swizzle: one
// warp's block of outputs (32 tokens x 32 columns, 64-byte rows) per store.
int encode_tokens_map_32(CUtensorMap* map, const void* base, int64_t T, int64_t H, int64_t D) {
  auto fn = encode_fn();
  if (!fn) return GDN_ERR_CUDA;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(T)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(D * 2), static_cast<cuuint64_t>(H * D * 2)};
  cuuint32_t box[3] = {32, 1, 32};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? GDN_OK : GDN_ERR_CUDA;
}

int encode_tiles_map_f16(CUtensorMap* map, const void* base, int64_t rows, int64_t cols) {
  auto fn = encode_fn();
  if (!fn) return GDN_ERR_CUDA;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols * 2)};
  cuuint32_t box[2] = {64, 64};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? GDN_OK : GDN_ERR_CUDA;
}

}  // namespace gdn_host

extern "C" const char* gdn_status_string(int status) {
  switch (status) {
    case GDN_OK:
      return "ok";
    case GDN_ERR_INVALID_ARGUMENT:
      return "invalid argument (null pointer, bad scalar or misaligned buffer)";
    case GDN_ERR_UNSUPPORTED:
      return "unsupported shape, dtype or device (K and V must be 128; sm_103a required)";
    case GDN_ERR_CUDA:
      return "a CUDA launch or driver call failed";
    default:
      return "unknown status";
  }
}
