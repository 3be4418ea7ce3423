// Host-side helpers shared by the CUDA entry points: device checks, TMA
// tensor-map encoding through the driver entry point (no link-time libcuda
// dependency), launch error mapping.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <mutex>
#include <utility>
#include <vector>

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

// Looked up once (thread-safe static initialisation).
inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
  }();
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

// Unique id of the CUDA context the calling thread's runtime calls act on
// (the device's primary context unless the caller made another one current).
// Ids are never reused within a process, so a context created after
// cudaDeviceReset, or another context on the same device, gets a new one.
// Returns false if no context is current or the driver cannot be asked.
inline bool current_context_id(unsigned long long* id) {
  static const auto fns = [] {
    void* get = nullptr;
    void* gid = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &get, 4000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      get = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &gid, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      gid = nullptr;
    return std::make_pair(reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(get), reinterpret_cast<PFN_cuCtxGetId_v12000>(gid));
  }();
  if (!fns.first || !fns.second) return false;
  CUcontext ctx = nullptr;
  if (fns.first(&ctx) != CUDA_SUCCESS || !ctx) return false;
  return fns.second(ctx, id) == CUDA_SUCCESS;
}

// A value set up once per CUDA context: kernel attributes such as the
// dynamic shared-memory limit belong to the context (one per device for the
// runtime's primary contexts), so a process that drives several GPUs, or
// recreates a context, has to set them again there.  Thread-safe.
template <typename T>
class PerContext {
 public:
  // The value for the current context, made by make(&value) -> status on
  // first use there.  make runs with the lock held; it may be a runtime call
  // that itself initialises the context, so the context is looked up after it.
  template <typename Make>
  int get(T* out, Make make) {
    unsigned long long id = 0;
    std::lock_guard<std::mutex> lock(mu_);
    if (current_context_id(&id))
      for (const auto& e : done_)
        if (e.first == id) {
          *out = e.second;
          return TPK_OK;
        }
    T v{};
    const int st = make(&v);
    if (st != TPK_OK) return st;
    if (current_context_id(&id)) done_.emplace_back(id, v);
    *out = v;
    return TPK_OK;
  }

 private:
  std::mutex mu_;
  std::vector<std::pair<unsigned long long, T>> done_;
};

// Raise a kernel's dynamic shared-memory limit to `bytes`, once per context.
template <typename Kern>
int set_smem_once(PerContext<int>& rec, Kern kern, size_t bytes) {
  int unused = 0;
  return rec.get(&unused, [&](int*) {
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes)) ==
                   cudaSuccess
               ? TPK_OK
               : TPK_E_CUDA;
  });
}

inline int num_sms() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

}  // namespace tpk
