// Moving per-token data between raw order and the packed (forwarded) layout.
//
// Gather ("Prefix Tree Packing in ART", section "Metadata space first": once a
// row's leaves are fixed, one pass slices token ids, logprobs, advantages and
// other per-token payloads into the packed tensors): each forwarded position
// takes the row of its owner, the lowest raw token mapping to it.
//
// Sum (the transpose of the raw-order scatter of "TRL Tree Packing for
// AsyncGRPO", section "How tree packing works", O_raw[r] = O[token_index[r]]):
// each forwarded position receives the sum of the rows of every raw token that
// maps to it -- how raw-order output gradients reach the packed layout.  The
// raw tokens of a position are the plan's CSR fwd_raw[fwd_raw_begin[f] ..
// fwd_raw_begin[f+1]), ascending, so the sums always run in the same order.
//
// Both are HBM-bound copies: 16-byte accesses wherever the row allows,
// consecutive threads on consecutive bytes of a row.
#include <cuda_bf16.h>

#include "common.cuh"

namespace tpk {
namespace {

constexpr int kThreads = 256;

// dst[f, c] = src[owner(f), c] over V-sized chunks c of rows of vpr chunks;
// one thread per chunk, a row's chunks on consecutive threads.
template <typename V>
__global__ void __launch_bounds__(kThreads) gather_kernel(const int32_t* __restrict__ begin,
                                                          const int32_t* __restrict__ raw, int64_t F,
                                                          const V* __restrict__ src, V* __restrict__ dst,
                                                          int64_t vpr) {
  const int64_t n = F * vpr;
  const int64_t step = static_cast<int64_t>(gridDim.x) * kThreads;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; i < n; i += step) {
    const int64_t f = i / vpr, c = i - f * vpr;
    const int64_t r = __ldg(raw + __ldg(begin + f));
    dst[i] = __ldg(src + r * vpr + c);
  }
}

__device__ __forceinline__ void add_bf16x8(float (&acc)[8], const uint4 v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    acc[2 * j] += __uint_as_float(w[j] << 16);
    acc[2 * j + 1] += __uint_as_float(w[j] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ uint32_t bf16x2_bits(float lo, float hi) {
  const __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&b);
}

// One warp per forwarded row; each lane owns 16-byte chunks (8 bf16) of the
// row and adds the raw rows in ascending raw order, starting from the first
// (a position with one raw token is copied bit for bit).  A lane takes kU
// chunks 32 apart at a time and issues their loads together, so each warp
// keeps kU * 512 bytes in flight per raw row: with one load per lane the
// resident warps held too few bytes in flight to cover HBM latency.
constexpr int kU = 4;

__global__ void __launch_bounds__(kThreads) sum_rows_kernel(const int32_t* __restrict__ begin,
                                                            const int32_t* __restrict__ raw, int64_t F,
                                                            const uint4* __restrict__ src, uint4* __restrict__ dst,
                                                            int vpr) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (kThreads / 32);
  for (int64_t f = static_cast<int64_t>(blockIdx.x) * (kThreads / 32) + (threadIdx.x >> 5); f < F; f += warps) {
    const int b = __ldg(begin + f), e = __ldg(begin + f + 1);
    const uint4* s0 = src + static_cast<int64_t>(__ldg(raw + b)) * vpr;
    uint4* d = dst + f * vpr;
    for (int c0 = lane; c0 < vpr; c0 += 32 * kU) {
      uint4 v[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u)
        if (c0 + 32 * u < vpr) v[u] = __ldg(s0 + c0 + 32 * u);
      if (e - b == 1) {
#pragma unroll
        for (int u = 0; u < kU; ++u)
          if (c0 + 32 * u < vpr) d[c0 + 32 * u] = v[u];
        continue;
      }
      float acc[kU][8];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          acc[u][2 * j] = __uint_as_float(w[j] << 16);
          acc[u][2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
        }
      }
      for (int k = b + 1; k < e; ++k) {
        const uint4* sk = src + static_cast<int64_t>(__ldg(raw + k)) * vpr;
#pragma unroll
        for (int u = 0; u < kU; ++u)
          if (c0 + 32 * u < vpr) v[u] = __ldg(sk + c0 + 32 * u);
#pragma unroll
        for (int u = 0; u < kU; ++u) add_bf16x8(acc[u], v[u]);
      }
#pragma unroll
      for (int u = 0; u < kU; ++u)
        if (c0 + 32 * u < vpr)
          d[c0 + 32 * u] = make_uint4(bf16x2_bits(acc[u][0], acc[u][1]), bf16x2_bits(acc[u][2], acc[u][3]),
                                      bf16x2_bits(acc[u][4], acc[u][5]), bf16x2_bits(acc[u][6], acc[u][7]));
    }
  }
}

// lse_dst[h, f] = sum of lse_src[h, r] over the raw tokens r of f (ascending);
// one thread per output element, coalesced writes.
__global__ void __launch_bounds__(kThreads) sum_lse_kernel(const int32_t* __restrict__ begin,
                                                           const int32_t* __restrict__ raw, int64_t F, int64_t R,
                                                           const float* __restrict__ src, float* __restrict__ dst,
                                                           int H) {
  const int64_t n = F * H;
  const int64_t step = static_cast<int64_t>(gridDim.x) * kThreads;
  for (int64_t idx = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; idx < n; idx += step) {
    const int64_t h = idx / F, f = idx % F;
    const int b = __ldg(begin + f), e = __ldg(begin + f + 1);
    const float* s = src + h * R;
    float acc = __ldg(s + __ldg(raw + b));
    for (int k = b + 1; k < e; ++k) acc += __ldg(s + __ldg(raw + k));
    dst[idx] = acc;
  }
}

int64_t grid_for(int64_t work, int64_t per_block) {
  int64_t blocks = (work + per_block - 1) / per_block;
  const int64_t cap = int64_t{num_sms()} * 16;
  if (blocks > cap) blocks = cap;
  return blocks < 1 ? 1 : blocks;
}

}  // namespace
}  // namespace tpk

extern "C" int tpk_gather_to_forwarded(const int32_t* fwd_raw_begin, const int32_t* fwd_raw, int64_t F, int64_t R,
                                       const void* src, void* dst, int64_t row_bytes, void* stream) {
  using namespace tpk;
  if (!fwd_raw_begin || !fwd_raw || !src || !dst || F < 0 || R < 0 || row_bytes <= 0) return TPK_E_ARG;
  if (F > R) return TPK_E_ARG;   // every forwarded position has at least one raw token
  if (F == 0) return TPK_OK;
  int st = check_device();
  if (st != TPK_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const uintptr_t al = reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst);
  if (row_bytes % 16 == 0 && al % 16 == 0) {
    const int64_t vpr = row_bytes / 16;
    gather_kernel<uint4><<<static_cast<unsigned>(grid_for(F * vpr, kThreads)), kThreads, 0, s>>>(
        fwd_raw_begin, fwd_raw, F, static_cast<const uint4*>(src), static_cast<uint4*>(dst), vpr);
  } else if (row_bytes % 4 == 0 && al % 4 == 0) {
    const int64_t vpr = row_bytes / 4;
    gather_kernel<uint32_t><<<static_cast<unsigned>(grid_for(F * vpr, kThreads)), kThreads, 0, s>>>(
        fwd_raw_begin, fwd_raw, F, static_cast<const uint32_t*>(src), static_cast<uint32_t*>(dst), vpr);
  } else {
    gather_kernel<uint8_t><<<static_cast<unsigned>(grid_for(F * row_bytes, kThreads)), kThreads, 0, s>>>(
        fwd_raw_begin, fwd_raw, F, static_cast<const uint8_t*>(src), static_cast<uint8_t*>(dst), row_bytes);
  }
  return cuda_status(cudaGetLastError());
}

extern "C" int tpk_sum_to_forwarded(const int32_t* fwd_raw_begin, const int32_t* fwd_raw, int64_t F, int64_t R,
                                    const void* src, void* dst, const float* lse_src, float* lse_dst, int32_t H,
                                    int32_t d, void* stream) {
  using namespace tpk;
  if (!fwd_raw_begin || !fwd_raw || F < 0 || R < 0 || H <= 0 || d <= 0) return TPK_E_ARG;
  if ((src == nullptr) != (dst == nullptr) || (lse_src == nullptr) != (lse_dst == nullptr)) return TPK_E_ARG;
  if (F > R) return TPK_E_ARG;
  if (src && ((static_cast<int64_t>(H) * d * 2) % 16 ||
              (reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst)) % 16))
    return TPK_E_ARG;
  if (F == 0) return TPK_OK;
  int st = check_device();
  if (st != TPK_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (src) {
    const int vpr = static_cast<int>(static_cast<int64_t>(H) * d * 2 / 16);
    sum_rows_kernel<<<static_cast<unsigned>(grid_for(F, kThreads / 32)), kThreads, 0, s>>>(
        fwd_raw_begin, fwd_raw, F, static_cast<const uint4*>(src), static_cast<uint4*>(dst), vpr);
    st = cuda_status(cudaGetLastError());
    if (st != TPK_OK) return st;
  }
  if (lse_src) {
    sum_lse_kernel<<<static_cast<unsigned>(grid_for(F * H, kThreads)), kThreads, 0, s>>>(fwd_raw_begin, fwd_raw, F,
                                                                                         R, lse_src, lse_dst, H);
    st = cuda_status(cudaGetLastError());
  }
  return st;
}
