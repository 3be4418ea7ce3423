// RoPE at tree-depth positions ("DAG packing", section "Positions": the
// position id of a token is its depth, so every parent->child edge has
// relative distance 1 wherever the two tokens sit in the row).
//
// HBM-bound: each position's Q and K rows are read and written once.  A block
// takes kPosPerBlock positions; it first builds their d/2 (cos, sin) pairs in
// shared memory (shared by all heads of Q and K), then streams the rows with
// 16-byte accesses: a thread rotates 8 pairs (x_i, x_{i+d/2}).
// The angle depth * base^(-2i/d) is reduced to a fraction of a turn in fp64
// (exact for depths < 2^31), then evaluated with sincospif in fp32.
#include <cuda_bf16.h>

#include "common.cuh"

namespace tpk {
namespace {

constexpr int kPosPerBlock = 4;
constexpr int kThreads = 256;

struct Turns {
  double v[64];   // base^(-2i/d) / (2 pi), i < d/2
};

__global__ void __launch_bounds__(kThreads) rope_kernel(const __nv_bfloat16* q_in, const __nv_bfloat16* k_in,
                                                        __nv_bfloat16* q_out, __nv_bfloat16* k_out,
                                                        const int32_t* __restrict__ depth, int64_t F, int Hq, int Hkv,
                                                        int D, Turns turns, int inverse) {
  __shared__ float cs[kPosPerBlock][64];
  __shared__ float sn[kPosPerBlock][64];
  const int half = D / 2;
  const int64_t f0 = static_cast<int64_t>(blockIdx.x) * kPosPerBlock;
  for (int t = threadIdx.x; t < kPosPerBlock * half; t += blockDim.x) {
    const int p = t / half, i = t % half;
    const int64_t f = f0 + p;
    float c = 1.f, s = 0.f;
    if (f < F) {
      double x = static_cast<double>(__ldg(depth + f)) * turns.v[i];
      x -= rint(x);   // fraction of a turn in [-1/2, 1/2]
      sincospif(static_cast<float>(2.0 * x), &s, &c);
      if (inverse) s = -s;
    }
    cs[p][i] = c;
    sn[p][i] = s;
  }
  __syncthreads();
  const int chunks = D / 16;   // 8 pairs per chunk
  const int heads = Hq + Hkv;
  const int items = kPosPerBlock * heads * chunks;
  for (int it = threadIdx.x; it < items; it += blockDim.x) {
    const int p = it / (heads * chunks);
    const int rem = it % (heads * chunks);
    const int h = rem / chunks, c = rem % chunks;
    const int64_t f = f0 + p;
    if (f >= F) continue;
    const __nv_bfloat16* src;
    __nv_bfloat16* dst;
    if (h < Hq) {
      src = q_in + (f * Hq + h) * D;
      dst = q_out + (f * Hq + h) * D;
    } else {
      src = k_in + (f * Hkv + (h - Hq)) * D;
      dst = k_out + (f * Hkv + (h - Hq)) * D;
    }
    const int i0 = c * 8;
    uint4 ua = *reinterpret_cast<const uint4*>(src + i0);
    uint4 ub = *reinterpret_cast<const uint4*>(src + half + i0);
    __nv_bfloat16* a = reinterpret_cast<__nv_bfloat16*>(&ua);
    __nv_bfloat16* b = reinterpret_cast<__nv_bfloat16*>(&ub);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float x = __bfloat162float(a[j]), y = __bfloat162float(b[j]);
      const float cc = cs[p][i0 + j], ss = sn[p][i0 + j];
      a[j] = __float2bfloat16_rn(x * cc - y * ss);
      b[j] = __float2bfloat16_rn(x * ss + y * cc);
    }
    *reinterpret_cast<uint4*>(dst + i0) = ua;
    *reinterpret_cast<uint4*>(dst + half + i0) = ub;
  }
}

}  // namespace
}  // namespace tpk

extern "C" int tpk_rope_by_depth(const void* q_in, const void* k_in, void* q_out, void* k_out,
                                 const int32_t* depth, int64_t F, int32_t Hq, int32_t Hkv, int32_t d, double base,
                                 int32_t inverse, void* stream) {
  using namespace tpk;
  if (F < 0 || !depth || (d != 64 && d != 128) || Hq < 0 || Hkv < 0 || !(base > 1.0)) return TPK_E_ARG;
  if ((q_in == nullptr) != (q_out == nullptr) || (k_in == nullptr) != (k_out == nullptr)) return TPK_E_ARG;
  if ((q_in && Hq <= 0) || (k_in && Hkv <= 0)) return TPK_E_ARG;
  if ((reinterpret_cast<uintptr_t>(q_in) | reinterpret_cast<uintptr_t>(k_in) | reinterpret_cast<uintptr_t>(q_out) |
       reinterpret_cast<uintptr_t>(k_out)) % 16)
    return TPK_E_ARG;
  if (F == 0 || (!q_in && !k_in)) return TPK_OK;
  int st = check_device();
  if (st != TPK_OK) return st;
  Turns turns;
  const double two_pi = 6.283185307179586476925286766559;
  for (int i = 0; i < d / 2; ++i) turns.v[i] = pow(base, -2.0 * i / d) / two_pi;
  const int64_t blocks = (F + kPosPerBlock - 1) / kPosPerBlock;
  if (blocks > 0x7fffffff) return TPK_E_OVERFLOW;
  rope_kernel<<<static_cast<unsigned>(blocks), kThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const __nv_bfloat16*>(q_in), static_cast<const __nv_bfloat16*>(k_in),
      static_cast<__nv_bfloat16*>(q_out), static_cast<__nv_bfloat16*>(k_out), depth, F, q_in ? Hq : 0,
      k_in ? Hkv : 0, d, turns, inverse);
  return cuda_status(cudaGetLastError());
}
