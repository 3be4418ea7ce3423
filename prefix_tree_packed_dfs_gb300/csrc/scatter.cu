// Scatter forwarded outputs back to raw-token order through token_index
// ("TRL Tree Packing for AsyncGRPO", section "How tree packing works": the
// collator maps every trained token back to its original position).
//
// HBM-bound copy.  Rows are H*d bf16 (4-8 KB); one warp moves one raw row
// with 16-byte loads/stores, so each warp instruction moves 512 contiguous
// bytes.  Forwarded rows shared by several raw tokens are read several times
// (L2 usually hits, since sharers are close in raw order only within a group).
// LSE [H, F] -> [H, R]: one thread per output element, coalesced writes.
#include <cuda_bf16.h>

#include "common.cuh"

namespace tpk {
namespace {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads) scatter_rows_kernel(const int32_t* __restrict__ ti, int64_t R,
                                                                const uint4* __restrict__ src,
                                                                uint4* __restrict__ dst, int vec_per_row) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (kThreads / 32);
  for (int64_t r = static_cast<int64_t>(blockIdx.x) * (kThreads / 32) + (threadIdx.x >> 5); r < R; r += warps) {
    const int64_t f = __ldg(ti + r);
    const uint4* s = src + f * vec_per_row;
    uint4* d = dst + r * vec_per_row;
    for (int c = lane; c < vec_per_row; c += 32) d[c] = __ldg(s + c);
  }
}

__global__ void __launch_bounds__(kThreads) scatter_lse_kernel(const int32_t* __restrict__ ti, int64_t R, int64_t F,
                                                               const float* __restrict__ src,
                                                               float* __restrict__ dst, int H) {
  const int64_t n = R * H;
  for (int64_t idx = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; idx < n;
       idx += static_cast<int64_t>(gridDim.x) * kThreads) {
    const int64_t h = idx / R, r = idx % R;
    dst[idx] = __ldg(src + h * F + __ldg(ti + r));
  }
}

}  // namespace
}  // namespace tpk

extern "C" int tpk_scatter_token_index(const int32_t* token_index, int64_t R, int64_t F, const void* src, void* dst,
                                       const float* lse_src, float* lse_dst, int32_t H, int32_t d, void* stream) {
  using namespace tpk;
  if (!token_index || R < 0 || F < 0 || H <= 0 || d <= 0) return TPK_E_ARG;
  if ((src == nullptr) != (dst == nullptr) || (lse_src == nullptr) != (lse_dst == nullptr)) return TPK_E_ARG;
  if ((static_cast<int64_t>(H) * d * 2) % 16) return TPK_E_ARG;
  if ((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst)) % 16) return TPK_E_ARG;
  if (R == 0) return TPK_OK;
  int st = check_device();
  if (st != TPK_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int sms = num_sms();
  if (src) {
    const int vec = static_cast<int>(static_cast<int64_t>(H) * d * 2 / 16);
    int64_t blocks = (R + (kThreads / 32) - 1) / (kThreads / 32);
    if (blocks > int64_t{sms} * 16) blocks = int64_t{sms} * 16;
    scatter_rows_kernel<<<static_cast<unsigned>(blocks), kThreads, 0, s>>>(
        token_index, R, static_cast<const uint4*>(src), static_cast<uint4*>(dst), vec);
    st = cuda_status(cudaGetLastError());
    if (st != TPK_OK) return st;
  }
  if (lse_src) {
    int64_t blocks = (R * H + kThreads - 1) / kThreads;
    if (blocks > int64_t{sms} * 16) blocks = int64_t{sms} * 16;
    scatter_lse_kernel<<<static_cast<unsigned>(blocks), kThreads, 0, s>>>(token_index, R, F, lse_src, lse_dst, H);
    st = cuda_status(cudaGetLastError());
  }
  return st;
}
