// Gradients of the GDN token mixer over a packed prefix tree (sm_103a).
//
// "Prefix Tree Packing in ART", section "Token-mixing layers": a child
// segment starts from a broadcast of its parent's final state, so autograd
// sums the gradients of every child back into that state.  These kernels
// compute the same sums without autograd: the delta rule's state gradient
// is carried backwards along each segment instance and, at its first token,
// handed to the parent instance, which adds the gradients of all its
// children before walking its own chain backwards; the convolution's input
// gradient gathers over every position whose window holds it (its own
// descendants on every branch below it).
//
// Convolution backward.  y = silu(a), a[f] = sum_j w_j x[anc_{W-1-j}(f)].
// dx[f] = sum over the descendants f' of f within W-1 steps (f itself at 0)
// of w_{W-1-t} da[f'], da = dy silu'(a), t = depth(f') - depth(f); dw_j =
// sum_f da[f] x[anc_{W-1-j}(f)].  A thread owns one 8-channel group of a
// stream of positions, as in the forward, and walks f's subtree in preorder
// down to depth W-1 (subtree_end skips deeper parts), recomputing each
// descendant's a from its window (the path between f and it, then f's own
// ancestors).  dw is summed per stream into a partial row; a second kernel
// adds the partials in a fixed order (deterministic).
//
// Delta rule backward, per head (k^, q~ = scale q^ the normalised k, q):
//   S_t = a_t S_{t-1} + u_t k^_t^T,  u_t = b_t (v_t - a_t w_t),  w_t = S_{t-1} k^_t,  o_t = S_t q~_t.
// With D_t = dL/dS_t (all later tokens and o_t), y_t = D_t k^_t:
//   dq~_t = S_t^T do_t,        dv_t = b_t y_t,       db_t = (v_t - a_t w_t) . y_t,
//   dk^_t = D_t^T u_t - a_t b_t S_{t-1}^T y_t,
//   dg_t  = psi_t - b_t v_t . y_t,   psi_t = <D_t, S_t>,
//   D_{t-1} = a_t (D_t - b_t y_t k^_t^T) + do_{t-1} q~_{t-1}^T,
//   psi_{t-1} = dg_t + do_{t-1} . o_{t-1}   (so dg needs no S_{t-1}).
// Then through the normalisations: dk = (dk^ - k^ (k^ . dk^)) / |k|, the
// same for q with the scale.
// One CTA per (segment instance, head), levels deepest first.  Pass A runs
// the instance forward from its initial state (the forward's saved parent
// state, zero at a root), keeping u_t, w_t, 1/|k_t|, do_t . o_t and the
// state every kCk tokens (checkpoints) in level-local scratch.  Pass B walks
// back from the final state: S_{t-1} = (S_t - u_t k^_t^T) / a_t, restarted
// from the exact checkpoint at every kCk-token boundary; where the product
// of 1/a since the last exact state would pass kAmpLimit (strong decay,
// where the reversal loses accuracy) S_{t-1} is replayed from the
// checkpoint instead.  D starts as the sum of the children's initial-state
// gradients (ascending child order), plus nothing at a leaf.
//
// State layout: D x D, 256 threads = 16 row tiles x 16 column tiles; warp w
// holds row tiles 2w, 2w+1 (lanes 0-15 / 16-31), column tile = lane & 15,
// whose columns are every 16th 16-byte chunk starting at chunk lane & 15.
// Row contractions (S k, S q, D k) reduce over the 16 lanes of a half warp;
// column contractions (S^T do, D^T u, S^T y) reduce over the two half warps
// and then over the 8 warps through shared memory, once per round of kRT
// tokens.
#include <cuda_bf16.h>

#include <algorithm>

#include "common.cuh"
#include "plan_handle.h"
#include "ptx.cuh"

namespace tpk {
namespace {

__device__ __forceinline__ float lo_bf(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi_bf(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ uint32_t bf2(float a, float b) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// ------------------------------------------------------------ convolution
constexpr int kCvThreads = 256;
constexpr int kCvMaxW = 8;
constexpr int64_t kCvThreadCap = int64_t{1} << 20;

constexpr int kCvRunHost = 64;   // positions per run of the backward kernel (kCvRun)

int64_t conv_streams(int64_t F, int C) {
  const int64_t cpr = C / 4;   // channel groups of the backward kernel (kCh)
  return std::max<int64_t>(1, std::min<int64_t>((F + kCvRunHost - 1) / kCvRunHost, kCvThreadCap / cpr));
}

// silu'(a) = s (1 + a (1 - s)), s = 1 / (1 + e^-a)
__device__ __forceinline__ float dsilu(float a) {
  const float s = __fdividef(1.f, 1.f + __expf(-a));
  return s * (1.f + a * (1.f - s));
}

// 4 channels (8 bytes) per thread in the backward: its rings hold W
// values per channel, so this keeps them in registers
constexpr int kCh = 4;

__device__ __forceinline__ float bf_at(const uint2& r, int e) {
  const uint32_t word = e < 2 ? r.x : r.y;
  return (e & 1) ? hi_bf(word) : lo_bf(word);
}

// dx[f] by the general walk: f's subtree in preorder down to depth W-1
// (subtree_end skips deeper parts), each descendant's pre-activation
// recomputed from its window (the path between f and it, then f's own
// ancestors).  Used where a fork lies within W-1 steps below f.
template <int W>
__device__ __forceinline__ void conv_bwd_walk(const int32_t* __restrict__ parent, const int32_t* __restrict__ depth,
                                              const int32_t* __restrict__ subtree_end, const uint2* __restrict__ x,
                                              const float (&wr)[kCh * W], const uint2* __restrict__ dy, int64_t f,
                                              int cpr, int g, float (&dxa)[kCh]) {
  uint2 anc[W];
  {
    int64_t a = f;
#pragma unroll
    for (int i = 0; i < W; ++i) {
      anc[i] = a >= 0 ? __ldg(x + a * cpr + g) : make_uint2(0u, 0u);
      if (i + 1 < W) a = a >= 0 ? __ldg(parent + a) : -1;
    }
  }
#pragma unroll
  for (int e = 0; e < kCh; ++e) dxa[e] = 0.f;
  uint2 st[W];
#pragma unroll
  for (int i = 0; i < W; ++i) st[i] = anc[0];
  auto visit = [&](const int T, const int64_t node) {   // T constant after unrolling
    const uint2 dv = __ldg(dy + node * cpr + g);
#pragma unroll
    for (int e = 0; e < kCh; ++e) {
      float a = 0.f;
#pragma unroll
      for (int i = 0; i < W; ++i) a = fmaf(wr[e * W + (W - 1 - i)], bf_at(i <= T ? st[T - i] : anc[i - T], e), a);
      dxa[e] = fmaf(wr[e * W + (W - 1 - T)], bf_at(dv, e) * dsilu(a), dxa[e]);
    }
  };
  visit(0, f);
  const int32_t d0 = __ldg(depth + f);
  const int64_t end = __ldg(subtree_end + f);
  int64_t node = f + 1;
  while (node < end) {
    const int t = __ldg(depth + node) - d0;
    const uint2 xv = __ldg(x + node * cpr + g);
#pragma unroll
    for (int T = 1; T < W; ++T)
      if (T == t) {
        st[T] = xv;
        visit(T, node);
      }
    node = t < W - 1 ? node + 1 : static_cast<int64_t>(__ldg(subtree_end + node));
  }
}

constexpr int kCvRun = 64;   // positions per run

// A thread owns one group of kCh channels and walks runs of kCvRun
// positions (runs s, s + streams, ..), ascending.  At each position p it
// keeps p's window (x at p and its W-1 nearest ancestors: shifted in from
// p-1 where p's parent is p-1, else gathered through the parent array) and
// the last W values of da = dy silu'(a); dw takes da[p] times the window
// (positions of the run only), and dx[p-W+1] is complete once da[p] is known:
//   dx[f] = sum_t w_{W-1-t} da[f+t]
// wherever the positions below f form one chain for W-1 steps (every node
// on it has one child, the next position, until a leaf), which the kinds
// of f .. f+W-2 tell (leaf: subtree_end = n+1; one child: subtree_end[n+1]
// = subtree_end[n]).  Elsewhere (a fork within W-1 steps below f) the
// general walk above computes dx[f].  A run reads W-1 positions past its
// end (their da) and recomputes them: (W-1)/kCvRun extra work.
template <int W>
__global__ void __launch_bounds__(kCvThreads) gdn_conv_bwd_kernel(
    const int32_t* __restrict__ parent, const int32_t* __restrict__ depth, const int32_t* __restrict__ subtree_end,
    const uint2* __restrict__ x, const float* __restrict__ w, const uint2* __restrict__ dy, uint2* __restrict__ dx,
    float* __restrict__ dw_part, int64_t F, int C, int64_t streams) {
  const int cpr = C / kCh;
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * kCvThreads + threadIdx.x;
  if (tid >= streams * cpr) return;
  const int g = static_cast<int>(tid % cpr);
  const int64_t s = tid / cpr;
  float wr[kCh * W];   // channel kCh g + e, tap j at wr[e * W + j]
  {
    const float4* w4 = reinterpret_cast<const float4*>(w + static_cast<int64_t>(g) * kCh * W);
#pragma unroll
    for (int i = 0; i < kCh * W / 4; ++i) {
      const float4 v = __ldg(w4 + i);
      wr[4 * i] = v.x;
      wr[4 * i + 1] = v.y;
      wr[4 * i + 2] = v.z;
      wr[4 * i + 3] = v.w;
    }
  }
  float dwa[kCh * W];
#pragma unroll
  for (int i = 0; i < kCh * W; ++i) dwa[i] = 0.f;
  const int64_t n_runs = (F + kCvRun - 1) / kCvRun;
  for (int64_t run = s; run < n_runs; run += streams) {
    const int64_t f0 = run * kCvRun, f1 = min(f0 + kCvRun, F);
    uint2 win[W];          // p's window: win[i] = x at p's i-th ancestor
    float da[W][kCh];      // da[W-1] at p, da[W-1-i] at p - i
    int kind[W];           // kind[W-1-i] of position p - 1 - i: 0 leaf, 1 one child, 2 fork
#pragma unroll
    for (int i = 0; i < W; ++i) {
      kind[i] = 0;
      win[i] = make_uint2(0u, 0u);
#pragma unroll
      for (int e = 0; e < kCh; ++e) da[i][e] = 0.f;
    }
    int32_t se_prev = 0;
    for (int64_t p = f0; p < f1 + W - 1; ++p) {
#pragma unroll
      for (int i = 0; i + 1 < W; ++i) {
        kind[i] = kind[i + 1];
#pragma unroll
        for (int e = 0; e < kCh; ++e) da[i][e] = da[i + 1][e];
      }
      if (p < F) {
        const int32_t par = __ldg(parent + p);
        const int32_t se = __ldg(subtree_end + p);
        const uint2 xp = __ldg(x + p * cpr + g);
        const uint2 dv = __ldg(dy + p * cpr + g);
        if (p > f0 && par == p - 1) {
#pragma unroll
          for (int i = W - 1; i > 0; --i) win[i] = win[i - 1];
        } else {
          int64_t a = par;
#pragma unroll
          for (int i = 1; i < W; ++i) {
            win[i] = a >= 0 ? __ldg(x + a * cpr + g) : make_uint2(0u, 0u);
            if (i + 1 < W) a = a >= 0 ? __ldg(parent + a) : -1;
          }
        }
        win[0] = xp;
#pragma unroll
        for (int e = 0; e < kCh; ++e) {
          float a = 0.f;
#pragma unroll
          for (int i = 0; i < W; ++i) a = fmaf(wr[e * W + (W - 1 - i)], bf_at(win[i], e), a);
          const float d = bf_at(dv, e) * dsilu(a);
          da[W - 1][e] = d;
          if (p < f1) {
#pragma unroll
            for (int i = 0; i < W; ++i) dwa[e * W + (W - 1 - i)] = fmaf(d, bf_at(win[i], e), dwa[e * W + (W - 1 - i)]);
          }
        }
        // the kind of p - 1, now that subtree_end[p] is known
        if (p > f0) kind[W - 1] = se_prev == p ? 0 : (se == se_prev ? 1 : 2);
        se_prev = se;
      } else {
#pragma unroll
        for (int e = 0; e < kCh; ++e) da[W - 1][e] = 0.f;
        kind[W - 1] = 0;   // past the end: F - 1 is a leaf
      }
      const int64_t f = p - (W - 1);
      if (f >= f0) {
        float acc[kCh];
        bool alive = true, fork = false;
#pragma unroll
        for (int e = 0; e < kCh; ++e) acc[e] = wr[e * W + (W - 1)] * da[0][e];
#pragma unroll
        for (int t = 1; t < W; ++t) {
          // the kind of f + t - 1 is kind[t] (kind[W-1] is p - 1 = f + W - 2)
          const int kd = kind[t];
          if (alive && kd == 2) fork = true;
          alive = alive && kd == 1;
          if (alive) {
#pragma unroll
            for (int e = 0; e < kCh; ++e) acc[e] = fmaf(wr[e * W + (W - 1 - t)], da[t][e], acc[e]);
          }
        }
        if (fork) conv_bwd_walk<W>(parent, depth, subtree_end, x, wr, dy, f, cpr, g, acc);
        dx[f * cpr + g] = make_uint2(bf2(acc[0], acc[1]), bf2(acc[2], acc[3]));
      }
    }
  }
  float* dst = dw_part + (s * C + static_cast<int64_t>(g) * kCh) * W;
#pragma unroll
  for (int i = 0; i < kCh * W; ++i) dst[i] = dwa[i];
}

// dw[c, j] = sum over streams of the partials, in stream order
__global__ void gdn_dw_reduce_kernel(const float* __restrict__ part, float* __restrict__ dw, int64_t n, int64_t streams) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n) return;
  float acc = 0.f;
  for (int64_t s = 0; s < streams; ++s) acc += __ldg(part + s * n + i);
  dw[i] = acc;
}

template <int W>
void launch_conv_bwd(const int32_t* par, const int32_t* dep, const int32_t* sub, const void* x, const float* w,
                     const void* dy, void* dx, float* part, int64_t F, int C, int64_t streams, cudaStream_t s) {
  const int64_t threads = streams * (C / kCh);
  gdn_conv_bwd_kernel<W><<<static_cast<unsigned>((threads + kCvThreads - 1) / kCvThreads), kCvThreads, 0, s>>>(
      par, dep, sub, static_cast<const uint2*>(x), w, static_cast<const uint2*>(dy), static_cast<uint2*>(dx), part, F,
      C, streams);
}

// ------------------------------------------------------------- delta rule
constexpr int kBT = 256;          // threads
constexpr int kRT = 16;           // tokens per staged round
constexpr int kCk = 32;           // checkpoint interval (tokens); a multiple of kRT
constexpr float kAmpLimit = 64.f; // largest growth of the reversal's error before a replay

struct GdnBwdParams {
  const __nv_bfloat16 *q, *k, *v, *dout;
  const float *g, *beta;
  __nv_bfloat16 *dq, *dk, *dv;
  float *dg, *dbeta;
  const int32_t *seg_start, *seg_len, *seg_parent, *seg_off;
  const float* state;   // the forward's final states [n_inst, H, D, D]
  float* G;             // initial-state gradients [n_inst, H, D, D]
  float* ck;            // checkpoints [slots, H, D, D] (level-local)
  float *U, *Wv;        // u_t, w_t [level tokens, H, D]
  float *dotv, *invk;   // do_t . o_t, 1/|k_t| [level tokens, H]
  int64_t ld_qk, ld_v, ld_dqk, ld_dv;
  int32_t H, inst0, next0, next1;
  float scale;
};

template <int D>
struct BwdSm {
  float k[kRT][D], q[kRT][D], v[kRT][D], dO[kRT][D], u[kRT][D], w[kRT][D], y[kRT][D];
  float part[kRT][8][2][D];   // per-warp column partials of dq~ and dk^
  float alpha[kRT], beta[kRT], ik[kRT], iq[kRT], vy[kRT], wy[kRT];
  float dot[kRT + 1];   // do . o of the round's tokens and of the token before it (pass B)
  float dgo[kRT];
  float dotp[kRT][8];
  float red[8];
};

template <int D>
__global__ void __launch_bounds__(kBT, 1) gdn_delta_bwd_kernel(const GdnBwdParams p) {
  constexpr int RT = D / 16, CT = D / 16;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  BwdSm<D>& sm = *reinterpret_cast<BwdSm<D>*>(smem_raw);
  const int inst = p.inst0 + static_cast<int>(blockIdx.x) / p.H;
  const int h = static_cast<int>(blockIdx.x) % p.H;
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int ct = lane & 15, rt = 2 * warp + (lane >> 4);
  const int r0 = rt * RT;
  const int start = __ldg(p.seg_start + inst), len = __ldg(p.seg_len + inst);
  const int par = __ldg(p.seg_parent + inst);
  const int off = __ldg(p.seg_off + inst);
  const int64_t slot0 = off / kCk + (inst - p.inst0);
  const int64_t HD = static_cast<int64_t>(p.H) * D;
  if (len <= 0) return;

  // S and D as packed fp32 pairs along the columns (two lanes per f32x2
  // instruction): S2[r][i] = columns colp(i), colp(i) + 1 of row r0 + r.  A
  // thread's columns are the 16-byte chunks ct, ct + 16, .. (4 columns
  // each), so the 16 column tiles of a half warp read one contiguous run of
  // a staged row and write one of the partial sums (no bank conflicts)
  constexpr int CP = CT / 2;
  auto colp = [&](int i) { return 4 * (ct + 16 * (i >> 1)) + 2 * (i & 1); };
  uint64_t S2[RT][CP], D2[RT][CP];
  auto tile_load = [&](uint64_t (&M)[RT][CP], const float* base) {   // base: [D][D] row-major
#pragma unroll
    for (int r = 0; r < RT; ++r)
#pragma unroll
      for (int i = 0; i < CP; i += 2) {
        const ulonglong2 v = *reinterpret_cast<const ulonglong2*>(base + (r0 + r) * D + colp(i));
        M[r][i] = v.x;
        M[r][i + 1] = v.y;
      }
  };
  auto tile_store = [&](const uint64_t (&M)[RT][CP], float* base) {
#pragma unroll
    for (int r = 0; r < RT; ++r)
#pragma unroll
      for (int i = 0; i < CP; i += 2)
        *reinterpret_cast<ulonglong2*>(base + (r0 + r) * D + colp(i)) = make_ulonglong2(M[r][i], M[r][i + 1]);
  };
  auto pair_sum = [](uint64_t v) {
    float lo, hi;
    ptx::unf2(v, lo, hi);
    return lo + hi;
  };
  // this thread's columns of a staged row as pairs
  auto row_pairs = [&](const float* rowp, uint64_t (&out)[CP]) {
#pragma unroll
    for (int i = 0; i < CP; i += 2) {
      const ulonglong2 v = ptx::lds128u(rowp + colp(i));
      out[i] = v.x;
      out[i + 1] = v.y;
    }
  };
  auto ck_ptr = [&](int64_t slot) { return p.ck + (slot * p.H + h) * static_cast<int64_t>(D) * D; };
  // sum over the 16 lanes of a half warp (the column tiles of a row tile)
  auto rowsum = [](float x) {
#pragma unroll
    for (int m = 1; m < 16; m <<= 1) x += __shfl_xor_sync(0xffffffffu, x, m);
    return x;
  };
  // stage tokens [j0, j0 + nt) of the instance: k^, q~ (fp32, normalised),
  // v, do, alpha, beta; with_uw: also u, w from the scratch
  auto stage = [&](int j0, int nt, bool with_uw) {
    constexpr int c8 = D / 8;
    for (int i = t; i < nt * 4 * c8; i += kBT) {
      const int j = i / (4 * c8), r = i % (4 * c8), which = r / c8, c = (r % c8) * 8;
      const int64_t f = start + j0 + j;
      const __nv_bfloat16* src = which == 0   ? p.k + f * p.ld_qk + h * D
                                 : which == 1 ? p.q + f * p.ld_qk + h * D
                                 : which == 2 ? p.v + f * p.ld_v + h * D
                                              : p.dout + f * HD + h * D;
      float* dst = which == 0 ? sm.k[j] : which == 1 ? sm.q[j] : which == 2 ? sm.v[j] : sm.dO[j];
      const uint4 raw = __ldg(reinterpret_cast<const uint4*>(src + c));
      const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        dst[c + 2 * a] = lo_bf(w4[a]);
        dst[c + 2 * a + 1] = hi_bf(w4[a]);
      }
    }
    if (with_uw) {
      for (int i = t; i < nt * 2 * (D / 4); i += kBT) {
        const int j = i / (2 * (D / 4)), r = i % (2 * (D / 4)), which = r / (D / 4), c = (r % (D / 4)) * 4;
        const int64_t tok = off + j0 + j;
        const float* src = (which == 0 ? p.U : p.Wv) + tok * HD + h * D + c;
        *reinterpret_cast<float4*>((which == 0 ? sm.u[j] : sm.w[j]) + c) = *reinterpret_cast<const float4*>(src);
      }
    }
    if (t < nt) {
      const int64_t f = start + j0 + t;
      sm.alpha[t] = __expf(__ldg(p.g + f * p.H + h));
      sm.beta[t] = __ldg(p.beta + f * p.H + h);
    }
    if (with_uw && t <= nt) {   // dot[i] = do . o of token j0 - 1 + i
      const int jj = j0 - 1 + t;
      sm.dot[t] = jj >= 0 ? p.dotv[(static_cast<int64_t>(off) + jj) * p.H + h] : 0.f;
    }
    __syncthreads();
    for (int j = warp; j < nt; j += kBT / 32) {
      float sk = 0.f, sq = 0.f;
      for (int c = lane; c < D; c += 32) {
        sk = fmaf(sm.k[j][c], sm.k[j][c], sk);
        sq = fmaf(sm.q[j][c], sm.q[j][c], sq);
      }
#pragma unroll
      for (int m = 16; m > 0; m >>= 1) {
        sk += __shfl_xor_sync(0xffffffffu, sk, m);
        sq += __shfl_xor_sync(0xffffffffu, sq, m);
      }
      const float ik = rsqrtf(sk), iq = rsqrtf(sq);
      const float iqs = iq * p.scale;
      for (int c = lane; c < D; c += 32) {
        sm.k[j][c] *= ik;
        sm.q[j][c] *= iqs;
      }
      if (lane == 0) {
        sm.ik[j] = ik;
        sm.iq[j] = iq;
      }
    }
    __syncthreads();
  };

  // ---------------- pass A: forward from the initial state, with scratch
  if (par >= 0) tile_load(S2, p.state + (static_cast<int64_t>(par) * p.H + h) * D * D);
  else {
#pragma unroll
    for (int r = 0; r < RT; ++r)
#pragma unroll
      for (int i = 0; i < CP; ++i) S2[r][i] = 0ull;
  }
  for (int j0 = 0; j0 < len; j0 += kRT) {
    const int nt = min(kRT, len - j0);
    stage(j0, nt, false);
    for (int j = 0; j < nt; ++j) {
      const int jj = j0 + j;
      if (jj % kCk == 0) tile_store(S2, ck_ptr(slot0 + jj / kCk));
      uint64_t k2[CP], q2[CP];
      row_pairs(sm.k[j], k2);
      row_pairs(sm.q[j], q2);
      const float a = sm.alpha[j], b = sm.beta[j];
      const uint64_t a2 = ptx::f2(a, a);
      float u[RT], wv[RT], o[RT];
#pragma unroll
      for (int r = 0; r < RT; ++r) {
        uint64_t acc = 0ull;
#pragma unroll
        for (int i = 0; i < CP; ++i) acc = ptx::fma2(S2[r][i], k2[i], acc);
        wv[r] = rowsum(pair_sum(acc));
        u[r] = b * (sm.v[j][r0 + r] - a * wv[r]);
      }
#pragma unroll
      for (int r = 0; r < RT; ++r) {
        const uint64_t u2 = ptx::f2(u[r], u[r]);
        uint64_t acc = 0ull;
#pragma unroll
        for (int i = 0; i < CP; ++i) {
          S2[r][i] = ptx::fma2(u2, k2[i], ptx::mul2(a2, S2[r][i]));
          acc = ptx::fma2(S2[r][i], q2[i], acc);
        }
        o[r] = rowsum(pair_sum(acc));
      }
      float dp = 0.f;
#pragma unroll
      for (int r = 0; r < RT; ++r) dp = fmaf(o[r], sm.dO[j][r0 + r], dp);
      dp += __shfl_xor_sync(0xffffffffu, dp, 16);
      if (lane == 0) sm.dotp[j][warp] = dp;
      // u and w rows of this row tile: lanes 0..RT-1 store u, RT..2RT-1 store w
      float su = 0.f;
#pragma unroll
      for (int r = 0; r < RT; ++r) {
        if (ct == r) su = u[r];
        if (ct == RT + r) su = wv[r];
      }
      const int64_t tok = off + jj;
      if (ct < 2 * RT) (ct < RT ? p.U : p.Wv)[tok * HD + h * D + r0 + (ct % RT)] = su;
    }
    __syncthreads();
    if (t < nt) {
      float s = 0.f;
#pragma unroll
      for (int w8 = 0; w8 < 8; ++w8) s += sm.dotp[t][w8];
      const int64_t tok = off + j0 + t;
      p.dotv[tok * p.H + h] = s;
      p.invk[tok * p.H + h] = sm.ik[t];
    }
  }
  // S = S_end.  Writes of pass A (U, W, dot, checkpoints) are read below by
  // other threads of this block.
  __syncthreads();

  // ---------------- pass B: backward
  // D = sum of the children's initial-state gradients (next level, one run)
  {
#pragma unroll
    for (int r = 0; r < RT; ++r)
#pragma unroll
      for (int i = 0; i < CP; ++i) D2[r][i] = 0ull;
    int lo = p.next0, hi = p.next1;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (__ldg(p.seg_parent + mid) < inst) lo = mid + 1;
      else hi = mid;
    }
    for (int c = lo; c < p.next1 && __ldg(p.seg_parent + c) == inst; ++c) {
      const float* src = p.G + (static_cast<int64_t>(c) * p.H + h) * D * D;
#pragma unroll
      for (int r = 0; r < RT; ++r)
#pragma unroll
        for (int i = 0; i < CP; i += 2) {
          const ulonglong2 v = *reinterpret_cast<const ulonglong2*>(src + (r0 + r) * D + colp(i));
          D2[r][i] = ptx::add2(D2[r][i], v.x);
          D2[r][i + 1] = ptx::add2(D2[r][i + 1], v.y);
        }
    }
  }
  // psi at the last token: <D_children, S_end> + do_end . o_end
  float psi = 0.f;
  {
    uint64_t s2 = 0ull;
#pragma unroll
    for (int r = 0; r < RT; ++r)
#pragma unroll
      for (int i = 0; i < CP; ++i) s2 = ptx::fma2(D2[r][i], S2[r][i], s2);
    float s = pair_sum(s2);
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) s += __shfl_xor_sync(0xffffffffu, s, m);
    if (lane == 0) sm.red[warp] = s;
    __syncthreads();
    if (t == 0) {
      float tot = 0.f;
#pragma unroll
      for (int w8 = 0; w8 < 8; ++w8) tot += sm.red[w8];
      psi = tot + p.dotv[(static_cast<int64_t>(off) + len - 1) * p.H + h];
    }
  }
  float amp = 1.f;
  for (int j0 = ((len - 1) / kRT) * kRT; j0 >= 0; j0 -= kRT) {
    const int nt = min(kRT, len - j0);
    __syncthreads();   // the previous round's epilogue is done with the staging
    stage(j0, nt, true);
    for (int j = nt - 1; j >= 0; --j) {
      const int jj = j0 + j;
      uint64_t k2[CP], q2[CP];
      row_pairs(sm.k[j], k2);
      row_pairs(sm.q[j], q2);
      float dor[RT], ur[RT];
#pragma unroll
      for (int r = 0; r < RT; ++r) {
        dor[r] = sm.dO[j][r0 + r];
        ur[r] = sm.u[j][r0 + r];
      }
      const float a = sm.alpha[j], b = sm.beta[j];
      const uint64_t a2 = ptx::f2(a, a);
      // D_t: add this token's output term
#pragma unroll
      for (int r = 0; r < RT; ++r) {
        const uint64_t d2 = ptx::f2(dor[r], dor[r]);
#pragma unroll
        for (int i = 0; i < CP; ++i) D2[r][i] = ptx::fma2(d2, q2[i], D2[r][i]);
      }
      float y[RT];
#pragma unroll
      for (int r = 0; r < RT; ++r) {
        uint64_t acc = 0ull;
#pragma unroll
        for (int i = 0; i < CP; ++i) acc = ptx::fma2(D2[r][i], k2[i], acc);
        y[r] = rowsum(pair_sum(acc));
      }
      uint64_t pq[CP], pk[CP];
#pragma unroll
      for (int i = 0; i < CP; ++i) {
        uint64_t aq = 0ull, ak = 0ull;
#pragma unroll
        for (int r = 0; r < RT; ++r) {
          aq = ptx::fma2(S2[r][i], ptx::f2(dor[r], dor[r]), aq);
          ak = ptx::fma2(D2[r][i], ptx::f2(ur[r], ur[r]), ak);
        }
        pq[i] = aq;
        pk[i] = ak;
      }
      // S_{t-1}
      if (jj % kCk == 0) {
        tile_load(S2, ck_ptr(slot0 + jj / kCk));
        amp = 1.f;
      } else {
        const float ia = 1.f / a;
        if (amp * ia > kAmpLimit) {
          // replay from the checkpoint of this block up to token jj - 1,
          // with the same operations as pass A
          const int jb = (jj / kCk) * kCk;
          tile_load(S2, ck_ptr(slot0 + jj / kCk));
          for (int m = jb; m < jj; ++m) {
            const int64_t f = start + m, tok = off + m;
            const float am = __expf(__ldg(p.g + f * p.H + h));
            const float ikm = p.invk[tok * p.H + h];
            const uint64_t am2 = ptx::f2(am, am);
            uint64_t km[CP];
#pragma unroll
            for (int i = 0; i < CP; ++i)
              km[i] = ptx::f2(__bfloat162float(p.k[f * p.ld_qk + h * D + colp(i)]) * ikm,
                              __bfloat162float(p.k[f * p.ld_qk + h * D + colp(i) + 1]) * ikm);
#pragma unroll
            for (int r = 0; r < RT; ++r) {
              const float um = p.U[tok * HD + h * D + r0 + r];
              const uint64_t um2 = ptx::f2(um, um);
#pragma unroll
              for (int i = 0; i < CP; ++i) S2[r][i] = ptx::fma2(um2, km[i], ptx::mul2(am2, S2[r][i]));
            }
          }
          amp = 1.f;
        } else {
          const uint64_t ia2 = ptx::f2(ia, ia);
#pragma unroll
          for (int r = 0; r < RT; ++r) {
            const uint64_t nu2 = ptx::f2(-ur[r], -ur[r]);
#pragma unroll
            for (int i = 0; i < CP; ++i) S2[r][i] = ptx::mul2(ptx::fma2(nu2, k2[i], S2[r][i]), ia2);
          }
          amp *= ia;
        }
      }
      {
        const float ab = a * b;
        const uint64_t nab2 = ptx::f2(-ab, -ab);
#pragma unroll
        for (int i = 0; i < CP; ++i) {
          uint64_t acc = 0ull;
#pragma unroll
          for (int r = 0; r < RT; ++r) acc = ptx::fma2(S2[r][i], ptx::f2(y[r], y[r]), acc);
          pk[i] = ptx::fma2(nab2, acc, pk[i]);
        }
      }
      // D_{t-1} without the previous token's output term
#pragma unroll
      for (int r = 0; r < RT; ++r) {
        const float by = b * y[r];
        const uint64_t nby2 = ptx::f2(-by, -by);
#pragma unroll
        for (int i = 0; i < CP; ++i) D2[r][i] = ptx::mul2(a2, ptx::fma2(nby2, k2[i], D2[r][i]));
      }
      // column partials of the two row tiles of this warp, then to shared
#pragma unroll
      for (int i = 0; i < CP; ++i) {
        pq[i] = ptx::add2(pq[i], __shfl_xor_sync(0xffffffffu, pq[i], 16));
        pk[i] = ptx::add2(pk[i], __shfl_xor_sync(0xffffffffu, pk[i], 16));
      }
      if (lane < 16) {
#pragma unroll
        for (int i = 0; i < CP; i += 2) {
          *reinterpret_cast<ulonglong2*>(&sm.part[j][warp][0][colp(i)]) = make_ulonglong2(pq[i], pq[i + 1]);
          *reinterpret_cast<ulonglong2*>(&sm.part[j][warp][1][colp(i)]) = make_ulonglong2(pk[i], pk[i + 1]);
        }
      }
      float sy = 0.f;
#pragma unroll
      for (int r = 0; r < RT; ++r)
        if (ct == r) sy = y[r];
      if (ct < RT) sm.y[j][r0 + ct] = sy;
    }
    __syncthreads();
    // epilogue: warp w finishes tokens w, w + 8 of the round
    for (int j = warp; j < nt; j += kBT / 32) {
      const int64_t f = start + j0 + j;
      float qd = 0.f, kd = 0.f, vy = 0.f, wy = 0.f;
      float gq[D / 32], gk[D / 32];
#pragma unroll
      for (int i = 0; i < D / 32; ++i) {
        const int c = lane + 32 * i;
        float sq = 0.f, sk = 0.f;
#pragma unroll
        for (int w8 = 0; w8 < 8; ++w8) {
          sq += sm.part[j][w8][0][c];
          sk += sm.part[j][w8][1][c];
        }
        gq[i] = sq;
        gk[i] = sk;
        qd = fmaf(sm.q[j][c], sq, qd);
        kd = fmaf(sm.k[j][c], sk, kd);
        vy = fmaf(sm.v[j][c], sm.y[j][c], vy);
        wy = fmaf(sm.w[j][c], sm.y[j][c], wy);
      }
#pragma unroll
      for (int m = 16; m > 0; m >>= 1) {
        qd += __shfl_xor_sync(0xffffffffu, qd, m);
        kd += __shfl_xor_sync(0xffffffffu, kd, m);
        vy += __shfl_xor_sync(0xffffffffu, vy, m);
        wy += __shfl_xor_sync(0xffffffffu, wy, m);
      }
      const float iq = sm.iq[j], ik = sm.ik[j], b = sm.beta[j];
      const float qs = qd / p.scale;
#pragma unroll
      for (int i = 0; i < D / 32; ++i) {
        const int c = lane + 32 * i;
        p.dq[f * p.ld_dqk + h * D + c] = __float2bfloat16_rn(iq * (p.scale * gq[i] - sm.q[j][c] * qs));
        p.dk[f * p.ld_dqk + h * D + c] = __float2bfloat16_rn(ik * (gk[i] - sm.k[j][c] * kd));
        p.dv[f * p.ld_dv + h * D + c] = __float2bfloat16_rn(b * sm.y[j][c]);
      }
      if (lane == 0) {
        sm.vy[j] = vy;
        sm.wy[j] = wy;
      }
    }
    __syncthreads();
    if (t == 0) {   // psi runs backwards through the round, in shared memory
      for (int j = nt - 1; j >= 0; --j) {
        const float dg = psi - sm.beta[j] * sm.vy[j];
        sm.dgo[j] = dg;
        psi = dg + sm.dot[j];   // + do . o of token j0 + j - 1 (0 before the first)
      }
    }
    __syncthreads();
    if (t < nt) {
      const int64_t f = start + j0 + t;
      p.dg[f * p.H + h] = sm.dgo[t];
      p.dbeta[f * p.H + h] = sm.vy[t] - sm.alpha[t] * sm.wy[t];
    }
  }
  // D = gradient of the initial state: the parent adds it to its own
  if (par >= 0) tile_store(D2, p.G + (static_cast<int64_t>(inst) * p.H + h) * D * D);
}

struct BwdScratch {
  size_t g_bytes, ck_bytes, uw_bytes, sc_bytes, total;
  int64_t max_tok, max_slots;
};

size_t al256(size_t x) { return (x + 255) & ~size_t(255); }

BwdScratch bwd_scratch(const Plan& P, int H, int D) {
  BwdScratch b{};
  const int n_levels = static_cast<int>(P.seg_level_begin.size()) - 1;
  for (int l = 0; l < n_levels; ++l) {
    int64_t tok = 0;
    for (int i = P.seg_level_begin[l]; i < P.seg_level_begin[l + 1]; ++i) tok += P.seg_len[i];
    const int64_t n = P.seg_level_begin[l + 1] - P.seg_level_begin[l];
    b.max_tok = std::max(b.max_tok, tok);
    b.max_slots = std::max(b.max_slots, tok / kCk + n + 1);
  }
  const size_t DD = static_cast<size_t>(D) * D * 4, hh = static_cast<size_t>(H);
  b.g_bytes = al256(P.seg_start.size() * hh * DD);
  b.ck_bytes = al256(static_cast<size_t>(b.max_slots) * hh * DD);
  b.uw_bytes = al256(static_cast<size_t>(b.max_tok) * hh * D * 4);
  b.sc_bytes = al256(static_cast<size_t>(b.max_tok) * hh * 4);
  b.total = b.g_bytes + b.ck_bytes + 2 * b.uw_bytes + 2 * b.sc_bytes;
  return b;
}

PerContext<int> g_smem_bwd64, g_smem_bwd128;

template <int D>
int launch_delta_bwd(const Plan& P, GdnBwdParams prm, cudaStream_t s) {
  const size_t smem = sizeof(BwdSm<D>);
  int st = set_smem_once(D == 128 ? g_smem_bwd128 : g_smem_bwd64, gdn_delta_bwd_kernel<D>, smem);
  if (st != TPK_OK) return st;
  const int n_levels = static_cast<int>(P.seg_level_begin.size()) - 1;
  for (int l = n_levels - 1; l >= 0; --l) {
    const int i0 = P.seg_level_begin[l], i1 = P.seg_level_begin[l + 1];
    const int64_t blocks = static_cast<int64_t>(i1 - i0) * prm.H;
    if (blocks <= 0) continue;
    if (blocks > 0x7fffffff) return TPK_E_OVERFLOW;
    prm.inst0 = i0;
    prm.next0 = i1;
    prm.next1 = l + 2 <= n_levels ? P.seg_level_begin[l + 2] : i1;
    gdn_delta_bwd_kernel<D><<<static_cast<unsigned>(blocks), kBT, smem, s>>>(prm);
    st = cuda_status(cudaGetLastError());
    if (st != TPK_OK) return st;
  }
  return TPK_OK;
}

}  // namespace
}  // namespace tpk

extern "C" size_t tpk_gdn_conv_bwd_workspace_bytes(const tpk_plan* plan, int32_t C, int32_t W) {
  using namespace tpk;
  if (!plan || C <= 0 || C % 8 || W < 1 || W > kCvMaxW) return 0;
  const int64_t F = plan->p.F;
  if (F == 0) return 0;
  return al256(static_cast<size_t>(conv_streams(F, C)) * static_cast<size_t>(C) * static_cast<size_t>(W) * 4);
}

extern "C" int tpk_gdn_conv_bwd(const tpk_plan* plan, const void* dev_image, const void* x, const float* w,
                                const void* dy, void* dx, float* dw, int32_t C, int32_t W, void* workspace,
                                size_t ws_bytes, void* stream) {
  using namespace tpk;
  if (!plan || !dev_image || !x || !w || !dy || !dx || !dw || C <= 0 || W < 1 || W > kCvMaxW) return TPK_E_ARG;
  if (C % 8 || (reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(dy) | reinterpret_cast<uintptr_t>(dx) |
                reinterpret_cast<uintptr_t>(w)) % 16)
    return TPK_E_ARG;
  const Plan& P = plan->p;
  if (P.F == 0) return TPK_OK;
  const size_t need = tpk_gdn_conv_bwd_workspace_bytes(plan, C, W);
  if (!workspace || ws_bytes < need || reinterpret_cast<uintptr_t>(workspace) % 256) return TPK_E_WORKSPACE;
  int st = check_device();
  if (st != TPK_OK) return st;
  const uint8_t* img = static_cast<const uint8_t*>(dev_image);
  const int32_t* par = reinterpret_cast<const int32_t*>(img + P.off_parent);
  const int32_t* dep = reinterpret_cast<const int32_t*>(img + P.off_depth);
  const int32_t* sub = reinterpret_cast<const int32_t*>(img + P.off_subtree_end);
  const int64_t streams = conv_streams(P.F, C);
  float* part = static_cast<float*>(workspace);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  switch (W) {
    case 1: launch_conv_bwd<1>(par, dep, sub, x, w, dy, dx, part, P.F, C, streams, s); break;
    case 2: launch_conv_bwd<2>(par, dep, sub, x, w, dy, dx, part, P.F, C, streams, s); break;
    case 3: launch_conv_bwd<3>(par, dep, sub, x, w, dy, dx, part, P.F, C, streams, s); break;
    case 4: launch_conv_bwd<4>(par, dep, sub, x, w, dy, dx, part, P.F, C, streams, s); break;
    case 5: launch_conv_bwd<5>(par, dep, sub, x, w, dy, dx, part, P.F, C, streams, s); break;
    case 6: launch_conv_bwd<6>(par, dep, sub, x, w, dy, dx, part, P.F, C, streams, s); break;
    case 7: launch_conv_bwd<7>(par, dep, sub, x, w, dy, dx, part, P.F, C, streams, s); break;
    default: launch_conv_bwd<8>(par, dep, sub, x, w, dy, dx, part, P.F, C, streams, s); break;
  }
  st = cuda_status(cudaGetLastError());
  if (st != TPK_OK) return st;
  const int64_t n = static_cast<int64_t>(C) * W;
  gdn_dw_reduce_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, s>>>(part, dw, n, streams);
  return cuda_status(cudaGetLastError());
}

extern "C" size_t tpk_gdn_bwd_workspace_bytes(const tpk_plan* plan, int32_t H, int32_t dk, int32_t dv) {
  using namespace tpk;
  if (!plan || H <= 0 || dk != dv || (dk != 64 && dk != 128)) return 0;
  if (plan->p.F == 0) return 0;
  return bwd_scratch(plan->p, H, dk).total;
}

extern "C" int tpk_gdn_delta_rule_bwd(const tpk_plan* plan, const void* dev_image, const void* q, const void* k,
                                      const void* v, int64_t ld_qk, int64_t ld_v, const float* g, const float* beta,
                                      const void* dout, void* dq, void* dk_, void* dv_, int64_t ld_dqk,
                                      int64_t ld_dv, float* dg, float* dbeta, int32_t H, int32_t dk, int32_t dv,
                                      float scale, const void* state, size_t state_bytes, void* workspace,
                                      size_t ws_bytes, void* stream) {
  using namespace tpk;
  if (!plan || !dev_image || !q || !k || !v || !g || !beta || !dout || !dq || !dk_ || !dv_ || !dg || !dbeta ||
      H <= 0 || !(scale > 0.f))
    return TPK_E_ARG;
  if (!((dk == 64 && dv == 64) || (dk == 128 && dv == 128))) return TPK_E_UNSUPPORTED;
  if (ld_qk < static_cast<int64_t>(H) * dk || ld_v < static_cast<int64_t>(H) * dv || ld_dqk < static_cast<int64_t>(H) * dk ||
      ld_dv < static_cast<int64_t>(H) * dv || ld_qk % 8 || ld_v % 8 || ld_dqk % 8 || ld_dv % 8)
    return TPK_E_ARG;
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v) |
       reinterpret_cast<uintptr_t>(dout)) % 16)
    return TPK_E_ARG;
  const Plan& P = plan->p;
  if (P.F == 0) return TPK_OK;
  if (!state || state_bytes < tpk_gdn_workspace_bytes(plan, H, dk, dv) || reinterpret_cast<uintptr_t>(state) % 16)
    return TPK_E_ARG;
  const BwdScratch b = bwd_scratch(P, H, dk);
  if (!workspace || ws_bytes < b.total || reinterpret_cast<uintptr_t>(workspace) % 256) return TPK_E_WORKSPACE;
  int st = check_device();
  if (st != TPK_OK) return st;
  const uint8_t* img = static_cast<const uint8_t*>(dev_image);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  GdnBwdParams prm;
  prm.q = static_cast<const __nv_bfloat16*>(q);
  prm.k = static_cast<const __nv_bfloat16*>(k);
  prm.v = static_cast<const __nv_bfloat16*>(v);
  prm.dout = static_cast<const __nv_bfloat16*>(dout);
  prm.g = g;
  prm.beta = beta;
  prm.dq = static_cast<__nv_bfloat16*>(dq);
  prm.dk = static_cast<__nv_bfloat16*>(dk_);
  prm.dv = static_cast<__nv_bfloat16*>(dv_);
  prm.dg = dg;
  prm.dbeta = dbeta;
  prm.seg_start = reinterpret_cast<const int32_t*>(img + P.off_seg_start);
  prm.seg_len = reinterpret_cast<const int32_t*>(img + P.off_seg_len);
  prm.seg_parent = reinterpret_cast<const int32_t*>(img + P.off_seg_parent);
  prm.seg_off = reinterpret_cast<const int32_t*>(img + P.off_seg_off);
  prm.state = static_cast<const float*>(state);
  prm.G = reinterpret_cast<float*>(ws);
  prm.ck = reinterpret_cast<float*>(ws + b.g_bytes);
  prm.U = reinterpret_cast<float*>(ws + b.g_bytes + b.ck_bytes);
  prm.Wv = reinterpret_cast<float*>(ws + b.g_bytes + b.ck_bytes + b.uw_bytes);
  prm.dotv = reinterpret_cast<float*>(ws + b.g_bytes + b.ck_bytes + 2 * b.uw_bytes);
  prm.invk = reinterpret_cast<float*>(ws + b.g_bytes + b.ck_bytes + 2 * b.uw_bytes + b.sc_bytes);
  prm.ld_qk = ld_qk;
  prm.ld_v = ld_v;
  prm.ld_dqk = ld_dqk;
  prm.ld_dv = ld_dv;
  prm.H = H;
  prm.inst0 = prm.next0 = prm.next1 = 0;
  prm.scale = scale;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return dk == 128 ? launch_delta_bwd<128>(P, prm, s) : launch_delta_bwd<64>(P, prm, s);
}
