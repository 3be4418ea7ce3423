// Host-side helpers shared by the CUDA entry points: device checks, TMA
// tensor-map encoding through the driver entry point (no link-time libcuda
// dependency), launch error mapping.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>

#include "tpk.h"

namespace tpk {

// Upper bound on any single device-side wait (mbarrier phase).  A wait that
// exceeds it marks the CTA aborted, every role leaves its loop, TMEM is freed
// and the launch reports TPK_E_TIMEOUT through dev_err.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

inline int cuda_status(cudaError_t e) { return e == cudaSuccess ? TPK_OK : TPK_E_CUDA; }

// True when the current device is an sm_103 part (the only target).
inline int check_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return TPK_E_CUDA;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return TPK_E_CUDA;
  if (cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) return TPK_E_CUDA;
  if (major != 10 || minor != 3) return TPK_E_UNSUPPORTED;
  return TPK_OK;
}

inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// Tensor map over a token-major bf16 tensor [rows, heads, d]: dims (d, heads,
// rows), box (64, 1, box_rows), 128-byte swizzle.  One box = box_rows rows of
// 64 elements (128 bytes) of one head, the canonical SW128 operand tile.
inline int make_map_bf16(CUtensorMap* map, const void* base, int64_t rows, int heads, int d, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return TPK_E_CUDA;
  if (reinterpret_cast<uintptr_t>(base) % 16) return TPK_E_ARG;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(heads), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(heads) * d * 2};
  cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estride[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estride,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? TPK_OK : TPK_E_CUDA;
}

inline int num_sms() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

}  // namespace tpk
