// GDN (Gated DeltaNet) token mixing over a packed prefix tree (sm_103a).
//
// "Prefix Tree Packing in ART", section "Token-mixing layers": GDN is the
// one layer that needs more than a mask.  It is recurrent: a running state is
// threaded token by token along each root-to-leaf path, forked once per
// branch point and reset at every tree root; it runs as a short causal
// convolution followed by the gated delta rule, one pass per tree depth.
//
// Convolution.  A position's causal window is its own path: itself and its
// W-1 nearest ancestors (the parent array), zero above a root.  So the whole
// packed batch is one launch -- each thread gathers its window through the
// parent pointers -- rather than one varlen call per depth with its initial
// conv state carried from the parent: the same sums, read where they lie.
//
// Delta rule, per head (k and q L2-normalised, alpha = exp(g)):
//   S_t = alpha_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,   o_t = S_t (scale q_t)
// written as  w = S k;  u = beta (v - alpha w);  S <- alpha S + u k^T;  o = S (scale q).
// The plan lists segment instances (a segment placed in one row: a chain of
// positions) by tree level; level l is one launch, one CTA per (instance,
// head).  A CTA starts from its parent instance's final state (kept in the
// workspace, fp32) or from zero at a root, runs its chain token by token and,
// if the chain has children, stores its final state for them.  The state
// carries across any token, so a branch point needs no chunk alignment: the
// pages' ragged-tail replay (their delta-rule kernel forks only at 64-token
// chunk boundaries) has nothing to do here.
//
// State layout: DV rows x DK columns in registers, 256 threads: thread t owns
// row t / TPR (TPR = 256 / DV threads per row) and every TPR-th 16-byte chunk
// of its columns starting at chunk t % TPR, as packed fp32 pairs -- the TPR
// threads of a row read neighbouring chunks of k and q, so a warp's shared
// load is one contiguous run; S k and S q are partial dot products summed
// over the TPR threads of a row with shuffles.  Tokens are staged kT at a time into
// shared memory (fp32, k and q normalised, q pre-scaled) and read back with
// broadcast 16-byte loads; outputs are gathered there and written back as
// bf16 rows.  Work per token and head: 6 dk dv FLOP (S k, the update, S q)
// on the fp32 pipes.
#include <cuda_bf16.h>

#include <algorithm>

#include "common.cuh"
#include "plan_handle.h"
#include "ptx.cuh"

namespace tpk {
namespace {

constexpr int kConvThreads = 256;
constexpr int kMaxConvW = 8;

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ uint32_t pack2(float a, float b) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}
__device__ __forceinline__ float silu(float a) { return a / (1.f + __expf(-a)); }

// y[f, c] = silu(sum_j w[c, j] x[a_{W-1-j}(f), c]), a_0 = f, a_{t+1} = parent(a_t).
// A thread owns one group of 8 channels (C % 8 == 0, 16-byte aligned rows)
// and walks positions f = f0, f0 + stride, ..: its 8 x W weights are one
// contiguous 32W-byte run of w, loaded once into registers; consecutive
// threads take consecutive channel groups of the same position, so row
// loads and stores are coalesced.  Inside a segment a position's parent is
// the position before it, so the parents of f, f-1, .., f-W+2 are loaded
// together and a_t taken from them while the chain holds; only where it
// breaks (a segment start) is the next ancestor a dependent load.
template <int W>
__global__ void __launch_bounds__(kConvThreads) gdn_conv_kernel(const int32_t* __restrict__ parent,
                                                                const uint4* __restrict__ x,
                                                                const float* __restrict__ w, uint4* __restrict__ y,
                                                                int64_t F, int C) {
  const int cpr = C / 8;   // 16-byte chunks (channel groups) per row
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * kConvThreads + threadIdx.x;
  const int64_t threads = static_cast<int64_t>(gridDim.x) * kConvThreads;
  const int64_t streams = threads / cpr;   // positions walked in parallel
  if (tid >= streams * cpr) return;
  const int g = static_cast<int>(tid % cpr);
  float wr[8 * W];   // weight of channel 8g + e, tap j at wr[e * W + j]
  {
    const float4* w4 = reinterpret_cast<const float4*>(w + static_cast<int64_t>(g) * 8 * W);
#pragma unroll
    for (int i = 0; i < 2 * W; ++i) {
      const float4 v = __ldg(w4 + i);
      wr[4 * i] = v.x;
      wr[4 * i + 1] = v.y;
      wr[4 * i + 2] = v.z;
      wr[4 * i + 3] = v.w;
    }
  }
  for (int64_t f = tid / cpr; f < F; f += streams) {
    int64_t a[W];
    a[0] = f;
    if constexpr (W > 1) {
      int32_t pf[W - 1];
#pragma unroll
      for (int t = 0; t < W - 1; ++t) pf[t] = f - t >= 0 ? __ldg(parent + f - t) : -1;
#pragma unroll
      for (int t = 1; t < W; ++t) {
        const int64_t prev = a[t - 1];
        a[t] = prev < 0 ? -1 : (prev == f - (t - 1) ? pf[t - 1] : __ldg(parent + prev));
      }
    }
    uint4 xv[W];
#pragma unroll
    for (int t = 0; t < W; ++t) xv[t] = a[t] >= 0 ? __ldg(x + a[t] * cpr + g) : make_uint4(0u, 0u, 0u, 0u);
    float acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      float s = 0.f;
#pragma unroll
      for (int t = 0; t < W; ++t) {   // tap W-1-t reads the t-th ancestor
        const uint32_t word = (&xv[t].x)[e / 2];
        s = fmaf(wr[e * W + (W - 1 - t)], (e & 1) ? bf16_hi(word) : bf16_lo(word), s);
      }
      acc[e] = s;
    }
    y[f * cpr + g] = make_uint4(pack2(silu(acc[0]), silu(acc[1])), pack2(silu(acc[2]), silu(acc[3])),
                                pack2(silu(acc[4]), silu(acc[5])), pack2(silu(acc[6]), silu(acc[7])));
  }
}

template <int W>
void launch_conv(const int32_t* parent, const void* x, const float* w, void* y, int64_t F, int C, int64_t blocks,
                 cudaStream_t s) {
  gdn_conv_kernel<W><<<static_cast<unsigned>(blocks), kConvThreads, 0, s>>>(
      parent, static_cast<const uint4*>(x), w, static_cast<uint4*>(y), F, C);
}

constexpr int kDeltaThreads = 256;
constexpr int kT = 16;   // tokens staged per round

struct DeltaParams {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  const float* g;
  const float* beta;
  __nv_bfloat16* o;
  const int32_t* seg_start;
  const int32_t* seg_len;
  const int32_t* seg_parent;
  const int32_t* subtree_end;
  float* state;        // [n_instances, H, DV, DK] fp32
  int64_t ld_qk, ld_v; // row strides (elements) of q, k and of v
  int32_t H, inst0;    // heads; first instance of this level
  float scale;
};

template <int DK, int DV>
struct DeltaSmem {
  alignas(16) float k[kT][DK];
  alignas(16) float q[kT][DK];
  alignas(16) float v[kT][DV];
  alignas(16) float o[kT][DV];
  float alpha[kT], beta[kT];
};

// Sum of a value over the TPR threads of a state row (consecutive lanes).
template <int TPR>
__device__ __forceinline__ float row_sum(float x) {
#pragma unroll
  for (int m = 1; m < TPR; m <<= 1) x += __shfl_xor_sync(0xffffffffu, x, m);
  return x;
}

template <int DK, int DV>
__global__ void __launch_bounds__(kDeltaThreads, 1) gdn_delta_kernel(const DeltaParams p) {
  constexpr int TPR = kDeltaThreads / DV;   // threads per state row
  constexpr int NCH = DK / 4 / TPR;         // 16-byte column chunks per thread
  static_assert(TPR >= 1 && TPR <= 32 && NCH >= 1 && DK % (4 * TPR) == 0, "state layout");
  __shared__ DeltaSmem<DK, DV> sm;
  const int inst = p.inst0 + static_cast<int>(blockIdx.x) / p.H;
  const int h = static_cast<int>(blockIdx.x) % p.H;
  const int t = threadIdx.x;
  const int e = t / TPR;                    // state row (value dimension)
  const int tc = t % TPR;                   // this thread owns column chunks tc, tc + TPR, ..
  const int start = __ldg(p.seg_start + inst), len = __ldg(p.seg_len + inst);
  const int par = __ldg(p.seg_parent + inst);
  // column of chunk i of this thread
  auto col = [&](int i) { return 4 * (tc + i * TPR); };

  uint64_t S[2 * NCH];   // chunk i = columns col(i)..col(i)+3 as two packed pairs
  if (par >= 0) {
    const float* src = p.state + ((static_cast<int64_t>(par) * p.H + h) * DV + e) * DK;
#pragma unroll
    for (int i = 0; i < NCH; ++i) {
      const ulonglong2 x = *reinterpret_cast<const ulonglong2*>(src + col(i));
      S[2 * i] = x.x;
      S[2 * i + 1] = x.y;
    }
  } else {
#pragma unroll
    for (int i = 0; i < 2 * NCH; ++i) S[i] = 0ull;
  }

  const int warp = t >> 5, lane = t & 31;
  // Round r's inputs are loaded into registers while round r-1 runs its
  // recurrence (the loads' latency hides behind kT tokens of work), then
  // written to shared memory as fp32 at the start of round r.
  constexpr int kc = DK / 8, vc = DV / 8;           // 16-byte chunks of a token's k (or q), v
  constexpr int kChunks = kT * (2 * kc + vc);
  constexpr int kPer = (kChunks + kDeltaThreads - 1) / kDeltaThreads;
  uint4 pre[kPer];
  float pre_g = 0.f, pre_b = 0.f;
  // chunk i of a round: token i / (2kc + vc); k chunks, then q, then v
  auto chunk_src = [&](int r0, int i) -> const uint4* {
    const int j = i / (2 * kc + vc), r = i % (2 * kc + vc);
    const int64_t f = start + r0 + j;
    if (r < kc) return reinterpret_cast<const uint4*>(p.k + f * p.ld_qk + h * DK + r * 8);
    if (r < 2 * kc) return reinterpret_cast<const uint4*>(p.q + f * p.ld_qk + h * DK + (r - kc) * 8);
    return reinterpret_cast<const uint4*>(p.v + f * p.ld_v + h * DV + (r - 2 * kc) * 8);
  };
  auto fetch = [&](int r0) {
    const int nt = min(kT, len - r0);
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int i = t + u * kDeltaThreads;
      if (i < nt * (2 * kc + vc)) pre[u] = __ldg(chunk_src(r0, i));
    }
    if (t < nt) {
      const int64_t f = start + r0 + t;
      pre_g = __ldg(p.g + f * p.H + h);
      pre_b = __ldg(p.beta + f * p.H + h);
    }
  };
  auto stage = [&](int r0) {
    const int nt = min(kT, len - r0);
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int i = t + u * kDeltaThreads;
      if (i >= nt * (2 * kc + vc)) continue;
      const int j = i / (2 * kc + vc), r = i % (2 * kc + vc);
      float* dst = r < kc ? &sm.k[j][r * 8] : r < 2 * kc ? &sm.q[j][(r - kc) * 8] : &sm.v[j][(r - 2 * kc) * 8];
      const uint32_t w4[4] = {pre[u].x, pre[u].y, pre[u].z, pre[u].w};
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        dst[2 * a] = bf16_lo(w4[a]);
        dst[2 * a + 1] = bf16_hi(w4[a]);
      }
    }
    if (t < nt) {
      sm.alpha[t] = __expf(pre_g);
      sm.beta[t] = pre_b;
    }
  };
  if (len > 0) fetch(0);
  for (int r0 = 0; r0 < len; r0 += kT) {
    const int nt = min(kT, len - r0);
    __syncthreads();   // the previous round's recurrence and outputs are done
    stage(r0);
    if (r0 + kT < len) fetch(r0 + kT);
    __syncthreads();
    // L2-normalise k and q of each staged token (one warp per token), q scaled
    for (int j = warp; j < nt; j += kDeltaThreads / 32) {
      float sk = 0.f, sq = 0.f;
      for (int c = lane; c < DK; c += 32) {
        sk = fmaf(sm.k[j][c], sm.k[j][c], sk);
        sq = fmaf(sm.q[j][c], sm.q[j][c], sq);
      }
#pragma unroll
      for (int m = 16; m > 0; m >>= 1) {
        sk += __shfl_xor_sync(0xffffffffu, sk, m);
        sq += __shfl_xor_sync(0xffffffffu, sq, m);
      }
      const float ik = rsqrtf(sk), iq = rsqrtf(sq) * p.scale;
      for (int c = lane; c < DK; c += 32) {
        sm.k[j][c] *= ik;
        sm.q[j][c] *= iq;
      }
    }
    __syncthreads();
    // The recurrence over the staged tokens.  The TPR threads of a row read
    // neighbouring 16-byte chunks of k and q, so a warp's load is one
    // contiguous run (no bank conflicts); k is read once and kept in
    // registers for both of its uses.
    for (int j = 0; j < nt; ++j) {
      ulonglong2 kk[NCH];
      uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
      for (int i = 0; i < NCH; ++i) {
        kk[i] = ptx::lds128u(&sm.k[j][col(i)]);
        acc[(2 * i) & 3] = ptx::fma2(S[2 * i], kk[i].x, acc[(2 * i) & 3]);
        acc[(2 * i + 1) & 3] = ptx::fma2(S[2 * i + 1], kk[i].y, acc[(2 * i + 1) & 3]);
      }
      float a0, a1;
      ptx::unf2(ptx::add2(ptx::add2(acc[0], acc[1]), ptx::add2(acc[2], acc[3])), a0, a1);
      const float wv = row_sum<TPR>(a0 + a1);
      const float a = sm.alpha[j];
      const float u = sm.beta[j] * (sm.v[j][e] - a * wv);
      const uint64_t a2x = ptx::f2(a, a), u2x = ptx::f2(u, u);
      // S <- a S + u k^T, then o = S q
      uint64_t oacc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
      for (int i = 0; i < NCH; ++i) {
        const ulonglong2 y = ptx::lds128u(&sm.q[j][col(i)]);
        S[2 * i] = ptx::fma2(u2x, kk[i].x, ptx::mul2(a2x, S[2 * i]));
        S[2 * i + 1] = ptx::fma2(u2x, kk[i].y, ptx::mul2(a2x, S[2 * i + 1]));
        oacc[(2 * i) & 3] = ptx::fma2(S[2 * i], y.x, oacc[(2 * i) & 3]);
        oacc[(2 * i + 1) & 3] = ptx::fma2(S[2 * i + 1], y.y, oacc[(2 * i + 1) & 3]);
      }
      float o0, o1;
      ptx::unf2(ptx::add2(ptx::add2(oacc[0], oacc[1]), ptx::add2(oacc[2], oacc[3])), o0, o1);
      const float ov = row_sum<TPR>(o0 + o1);
      if (tc == 0) sm.o[j][e] = ov;
    }
    __syncthreads();
    // outputs of the round: nt rows of DV as bf16, 8 per thread-chunk
    for (int i = t; i < nt * vc; i += kDeltaThreads) {
      const int j = i / vc, c = (i % vc) * 8;
      const float* src = &sm.o[j][c];
      __nv_bfloat16* dst = p.o + (static_cast<int64_t>(start + r0 + j) * p.H + h) * DV + c;
      *reinterpret_cast<uint4*>(dst) = make_uint4(pack2(src[0], src[1]), pack2(src[2], src[3]),
                                                  pack2(src[4], src[5]), pack2(src[6], src[7]));
    }
  }
  // the final state, for the children of a chain that has any
  const bool has_children = len > 0 && __ldg(p.subtree_end + start + len - 1) > start + len;
  if (has_children) {
    float* dst = p.state + ((static_cast<int64_t>(inst) * p.H + h) * DV + e) * DK;
#pragma unroll
    for (int i = 0; i < NCH; ++i) *reinterpret_cast<ulonglong2*>(dst + col(i)) = make_ulonglong2(S[2 * i], S[2 * i + 1]);
  }
}

template <int DK, int DV>
int launch_levels(const Plan& P, DeltaParams prm, cudaStream_t s) {
  const int n_levels = static_cast<int>(P.seg_level_begin.size()) - 1;
  for (int l = 0; l < n_levels; ++l) {
    const int i0 = P.seg_level_begin[l], i1 = P.seg_level_begin[l + 1];
    const int64_t blocks = static_cast<int64_t>(i1 - i0) * prm.H;
    if (blocks <= 0) continue;
    if (blocks > 0x7fffffff) return TPK_E_OVERFLOW;
    prm.inst0 = i0;
    gdn_delta_kernel<DK, DV><<<static_cast<unsigned>(blocks), kDeltaThreads, 0, s>>>(prm);
    const int st = cuda_status(cudaGetLastError());
    if (st != TPK_OK) return st;
  }
  return TPK_OK;
}

}  // namespace
}  // namespace tpk

extern "C" int tpk_gdn_conv(const tpk_plan* plan, const void* dev_image, const void* x, const float* w, void* y,
                            int32_t C, int32_t W, void* stream) {
  using namespace tpk;
  if (!plan || !dev_image || !x || !w || !y || C <= 0 || W < 1 || W > kMaxConvW) return TPK_E_ARG;
  if (C % 8 || (reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y) | reinterpret_cast<uintptr_t>(w)) % 16)
    return TPK_E_ARG;
  const Plan& P = plan->p;
  if (P.F == 0) return TPK_OK;
  int st = check_device();
  if (st != TPK_OK) return st;
  // enough threads for every channel group and many positions in flight,
  // rounded to whole position streams
  const int64_t cpr = C / 8;
  int64_t threads = std::min<int64_t>(P.F * cpr, int64_t{num_sms()} * 2048);
  threads = std::max<int64_t>(cpr, threads / cpr * cpr);
  const int64_t blocks = (threads + kConvThreads - 1) / kConvThreads;
  const int32_t* par = reinterpret_cast<const int32_t*>(static_cast<const uint8_t*>(dev_image) + P.off_parent);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  switch (W) {
    case 1: launch_conv<1>(par, x, w, y, P.F, C, blocks, s); break;
    case 2: launch_conv<2>(par, x, w, y, P.F, C, blocks, s); break;
    case 3: launch_conv<3>(par, x, w, y, P.F, C, blocks, s); break;
    case 4: launch_conv<4>(par, x, w, y, P.F, C, blocks, s); break;
    case 5: launch_conv<5>(par, x, w, y, P.F, C, blocks, s); break;
    case 6: launch_conv<6>(par, x, w, y, P.F, C, blocks, s); break;
    case 7: launch_conv<7>(par, x, w, y, P.F, C, blocks, s); break;
    default: launch_conv<8>(par, x, w, y, P.F, C, blocks, s); break;
  }
  return cuda_status(cudaGetLastError());
}

extern "C" size_t tpk_gdn_workspace_bytes(const tpk_plan* plan, int32_t H, int32_t dk, int32_t dv) {
  if (!plan || H <= 0 || dk <= 0 || dv <= 0) return 0;
  return (plan->p.seg_start.size() * static_cast<size_t>(H) * static_cast<size_t>(dk) * static_cast<size_t>(dv) * 4 +
          255) & ~size_t(255);
}

extern "C" int tpk_gdn_delta_rule(const tpk_plan* plan, const void* dev_image, const void* q, const void* k,
                                  const void* v, int64_t ld_qk, int64_t ld_v, const float* g, const float* beta,
                                  void* o, int32_t H, int32_t dk, int32_t dv, float scale, void* workspace,
                                  size_t ws_bytes, void* stream) {
  using namespace tpk;
  if (!plan || !dev_image || !q || !k || !v || !g || !beta || !o || H <= 0 || !(scale > 0.f)) return TPK_E_ARG;
  if (!((dk == 64 && dv == 64) || (dk == 128 && dv == 128))) return TPK_E_UNSUPPORTED;
  if (ld_qk < static_cast<int64_t>(H) * dk || ld_v < static_cast<int64_t>(H) * dv || ld_qk % 8 || ld_v % 8)
    return TPK_E_ARG;
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v) |
       reinterpret_cast<uintptr_t>(o)) % 16)
    return TPK_E_ARG;
  const Plan& P = plan->p;
  if (P.F == 0) return TPK_OK;
  const size_t need = tpk_gdn_workspace_bytes(plan, H, dk, dv);
  if (!workspace || ws_bytes < need || reinterpret_cast<uintptr_t>(workspace) % 256) return TPK_E_WORKSPACE;
  int st = check_device();
  if (st != TPK_OK) return st;
  const uint8_t* img = static_cast<const uint8_t*>(dev_image);
  DeltaParams prm;
  prm.q = static_cast<const __nv_bfloat16*>(q);
  prm.k = static_cast<const __nv_bfloat16*>(k);
  prm.v = static_cast<const __nv_bfloat16*>(v);
  prm.g = g;
  prm.beta = beta;
  prm.o = static_cast<__nv_bfloat16*>(o);
  prm.seg_start = reinterpret_cast<const int32_t*>(img + P.off_seg_start);
  prm.seg_len = reinterpret_cast<const int32_t*>(img + P.off_seg_len);
  prm.seg_parent = reinterpret_cast<const int32_t*>(img + P.off_seg_parent);
  prm.subtree_end = reinterpret_cast<const int32_t*>(img + P.off_subtree_end);
  prm.state = static_cast<float*>(workspace);
  prm.ld_qk = ld_qk;
  prm.ld_v = ld_v;
  prm.H = H;
  prm.inst0 = 0;
  prm.scale = scale;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return dk == 128 ? launch_levels<128, 128>(P, prm, s) : launch_levels<64, 64>(P, prm, s);
}
