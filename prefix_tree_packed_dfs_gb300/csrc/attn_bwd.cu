// Tree attention backward on tcgen05 (sm_103a).
//
// Gradients of L = sum_{f,h} <dO[f,h], O[f,h]> for the forward of attn_fwd.cu
// (every query attends to itself and its ancestors, j <= i < subtree_end[j];
// "Prefix Tree Packing in ART", section "Token-mixing layers").  With
// P_ij = exp(scale q_i.k_j - LSE_i) on visible pairs (0 elsewhere),
// dP_ij = dO_i.v_j, D_i = dO_i.O_i and dS_ij = P_ij (dP_ij - D_i):
//   dV_j = sum_i P_ij dO_i,  dK_j = scale sum_i dS_ij q_i,  dQ_i = scale sum_j dS_ij k_j.
//
// Three launches, all deterministic (no atomics):
//  1. prep:      D[h,i] = dO_i . O_i (fp32, into the workspace).
//  2. key-major: one CTA per (128-key tile, KV head).  It walks the tile's
//     query blocks -- [k0, max subtree_end) of its keys, the only queries that
//     can see them -- for every query head of the group, and keeps dK, dV of
//     the tile in TMEM.  Per (query block, head):
//        S^T = K Q^T, dP^T = V dO^T            (tcgen05, operands from smem)
//        softmax warps: P^T, dS^T -> bf16, written back into TMEM over S^T, dP^T
//        dV += P^T dO, dK += dS^T Q            (A operand straight from TMEM)
//  3. query-major: one CTA per (128-query tile, query head), the forward's key
//     blocks:  S = Q K^T, dP = dO V^T, dS -> TMEM, dQ += dS K.
// Pass 3 recomputes S and dP (7 matrix products instead of 5) in exchange for
// a dQ that needs neither an fp32 accumulator nor atomics.
//
// Precision.  The fast mode feeds P and dS to their products as bf16, as a
// bf16 flash-attention backward does.  The precise mode splits each of them
// into a bf16 high part and the bf16 rounding of the remainder and multiplies
// both (one more product for each of dV, dK and dQ), so they enter with about
// 16 significant bits; the prep pass then also adds the forward's rounding
// residual of O (D = dO . (O + O_lo)).  In TMEM every 32-column part of a
// score tile holds its high half in the first 16 columns and its low half in
// the next 16, so a part's stores only touch columns its own loads have read.
// Inverse RoPE: with rope set, the dK and dQ epilogues rotate each fp32
// gradient row back by its depth's angle ("DAG packing", section
// "Positions") before the one bf16 rounding, giving gradients w.r.t. the
// un-rotated inputs without another pass over them.
//
// Warp roles in passes 2 and 3: warp 0 TMA producer, warp 1 MMA issuer and
// TMEM owner, warps 4-7 the 128 row threads (one TMEM lane each).  Waits are
// bounded as in the forward; a timeout sets *dev_err = TPK_E_TIMEOUT.
#include <cuda_bf16.h>

#include <cmath>

#include "common.cuh"
#include "plan_handle.h"
#include "ptx.cuh"

namespace tpk {
namespace {

constexpr int BT = 128;          // tile height (keys in pass 2, queries in pass 3)
constexpr int kBox = BT * 128;   // one 128-row x 64-element swizzled box
constexpr float kLog2e = 1.4426950408889634f;

struct BwdParams {
  // forward work list (pass 3)
  const int32_t* qt_q0;
  const int32_t* qt_nq;
  const int32_t* qt_kb_begin;
  const int2* kb;
  const int32_t* qt_order;
  // backward work list (pass 2)
  const int32_t* kt_k0;
  const int32_t* kt_nk;
  const int32_t* kt_qb_begin;
  const int2* qb;
  const int32_t* kt_order;
  const int32_t* subtree_end;
  const float* lse;     // [Hq, F]
  const float* dsum;    // [Hq, F]
  __nv_bfloat16* dq;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  int32_t F, Hq, Hkv, group_size;
  float scale, scale_log2;
  int32_t* err;
  // inverse RoPE in the dK / dQ epilogues (rope != 0): depth [F] and the
  // per-frequency turn factors base^(-2i/d) / (2 pi) as fp32 pairs hi + lo
  const int32_t* depth;
  int32_t rope;
  float rope_hi[64], rope_lo[64];
};

// ----------------------------------------------------------------- pass 1
// D[h, f] = dO[f, h, :] . O[f, h, :] in fp32.  A row of D bf16 is D/8
// 16-byte chunks; that many lanes share a row (two rows per warp at D = 128,
// four at D = 64) and add their partial dots with shuffles inside the group.
// With o_lo (the precise mode's rounding residual of O from the forward) the
// dot is taken with O + O_lo.
__global__ void __launch_bounds__(256) bwd_prep_kernel(const __nv_bfloat16* __restrict__ o,
                                                       const __nv_bfloat16* __restrict__ o_lo,
                                                       const __nv_bfloat16* __restrict__ dout,
                                                       float* __restrict__ dsum, int64_t F, int Hq, int D) {
  const int lane = threadIdx.x & 31;
  const int lpr = D / 8;            // lanes per row
  const int rpw = 32 / lpr;         // rows per warp step
  const int sub = lane / lpr, cl = lane % lpr;
  const int64_t n = F * Hq;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t w0 = (static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5)) * rpw; w0 < n;
       w0 += nwarps * rpw) {
    const int64_t w = w0 + sub;
    float acc = 0.f;
    if (w < n) {
      const uint4 a = __ldg(reinterpret_cast<const uint4*>(o + w * D) + cl);
      const uint4 b = __ldg(reinterpret_cast<const uint4*>(dout + w * D) + cl);
      const uint32_t x[4] = {a.x, a.y, a.z, a.w}, y[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        acc = fmaf(__uint_as_float(x[j] << 16), __uint_as_float(y[j] << 16), acc);
        acc = fmaf(__uint_as_float(x[j] & 0xFFFF0000u), __uint_as_float(y[j] & 0xFFFF0000u), acc);
      }
      if (o_lo) {
        const uint4 c = __ldg(reinterpret_cast<const uint4*>(o_lo + w * D) + cl);
        const uint32_t z[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          acc = fmaf(__uint_as_float(z[j] << 16), __uint_as_float(y[j] << 16), acc);
          acc = fmaf(__uint_as_float(z[j] & 0xFFFF0000u), __uint_as_float(y[j] & 0xFFFF0000u), acc);
        }
      }
    }
    for (int off = lpr / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (cl == 0 && w < n) dsum[(w % Hq) * F + w / Hq] = acc;
  }
}

// cos and sin of the RoPE angle of one frequency at depth p (p < 2^24, exact
// in fp32).  The angle in turns is p * t with t = base^(-2i/d) / (2 pi) given
// as an fp32 pair hi + lo: the product p * hi is split exactly with an fma,
// its whole turns dropped, the remainders added (the fraction of a turn to
// ~3e-8), and the hardware sine / cosine evaluated on the reduced angle,
// which lies in [-pi, pi].
__device__ __forceinline__ void rope_cs(float pf, float hi, float lo, float& c, float& s) {
  const float a = pf * hi;
  const float e = fmaf(pf, hi, -a);
  const float f = (a - rintf(a)) + fmaf(pf, lo, e);
  __sincosf(6.28318530717958647692f * f, &s, &c);
}

// Inverse rotation of W frequency pairs of one gradient row and their store:
// ua holds columns [f0, f0 + W) and ub columns [f0 + D/2, f0 + D/2 + W) (fp32
// TMEM words), scaled by mul; x' = x cos + y sin, y' = y cos - x sin.
template <int W>
__device__ __forceinline__ void store_rotated(__nv_bfloat16* row, int f0, int half_d, const uint32_t* ua,
                                              const uint32_t* ub, float mul, float pf, const BwdParams& p) {
  uint32_t pa[W / 2], pb[W / 2];
#pragma unroll
  for (int j = 0; j < W; j += 2) {
    float c0, s0, c1, s1;
    rope_cs(pf, p.rope_hi[f0 + j], p.rope_lo[f0 + j], c0, s0);
    rope_cs(pf, p.rope_hi[f0 + j + 1], p.rope_lo[f0 + j + 1], c1, s1);
    const float x0 = __uint_as_float(ua[j]) * mul, y0 = __uint_as_float(ub[j]) * mul;
    const float x1 = __uint_as_float(ua[j + 1]) * mul, y1 = __uint_as_float(ub[j + 1]) * mul;
    pa[j / 2] = ptx::pack_bf16x2(fmaf(x0, c0, y0 * s0), fmaf(x1, c1, y1 * s1));
    pb[j / 2] = ptx::pack_bf16x2(fmaf(y0, c0, -x0 * s0), fmaf(y1, c1, -x1 * s1));
  }
  uint4* da = reinterpret_cast<uint4*>(row + f0);
  uint4* db = reinterpret_cast<uint4*>(row + half_d + f0);
#pragma unroll
  for (int j = 0; j < W / 8; ++j) {
    da[j] = make_uint4(pa[4 * j], pa[4 * j + 1], pa[4 * j + 2], pa[4 * j + 3]);
    db[j] = make_uint4(pb[4 * j], pb[4 * j + 1], pb[4 * j + 2], pb[4 * j + 3]);
  }
}

// TMEM column of the bf16 A operand for the 16-row K-step kk of a 64-wide
// score tile: part kk/2 (32 rows) starts at column 32*(kk/2), its high half in
// the first 16 columns (8 per K-step), its low half 16 columns further.
__device__ __forceinline__ constexpr uint32_t a_col(int kk, bool lo) {
  return 32u * static_cast<uint32_t>(kk >> 1) + 8u * static_cast<uint32_t>(kk & 1) + (lo ? 16u : 0u);
}

// Row epilogue helper: 32 fp32 TMEM columns * mul -> 32 bf16 stored to dst.
__device__ __forceinline__ void store_row32(__nv_bfloat16* dst, const uint32_t (&u)[32], float mul) {
  uint32_t pk[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) pk[j] = ptx::pack_bf16x2(__uint_as_float(u[2 * j]) * mul, __uint_as_float(u[2 * j + 1]) * mul);
  uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int j = 0; j < 4; ++j) d4[j] = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
}

// ----------------------------------------------------------------- pass 2
// Key-major dK/dV.  Each step (query block, query head) is split into two
// 64-query halves that alternate between two TMEM slots, so the tensor cores
// run one half's products while a softmax warpgroup works on the other:
//   MMA order per step n:  S/dP(n, half 0) | dV/dK(n-1, half 1) | S/dP(n, half 1) | dV/dK(n, half 0)
// TMEM: slot h at [128h, 128h+128): S^T (64 cols) then dP^T (64 cols);
// dV at [256, 256+D), dK at [256+D, 256+2D).  P^T and dS^T (bf16) overwrite
// S^T and dP^T of their slot in two 32-query parts (columns 32c.., high
// halves first, low halves 16 columns on in the precise mode) that the
// softmax releases one after the other (p_part, p_full) so the first part's
// dV/dK products start early.  S^T and dP^T read K and V from
// shared memory: the two slots and dK, dV fill TMEM.
// Warps: 0 TMA producer, 1 MMA issuer + TMEM owner, 2 loads LSE*log2(e) and D
// of each step's 128 queries into shared memory, 4-7 softmax of half 0,
// 8-11 softmax of half 1.
constexpr int kHalf = 64;
constexpr int kStat = 4;   // row-term ring depth of the dK/dV pass
constexpr int kHalfBox = kHalf * 128;   // one 64-row x 64-element swizzled box

template <int D, int NH>
struct KVSmem {
  uint8_t k[D / 64][kBox];
  uint8_t v[D / 64][kBox];
  uint8_t q[NH][D / 64][kHalfBox];
  uint8_t dO[NH][D / 64][kHalfBox];
  alignas(16) float lse2[kStat][BT];   // -LSE * log2(e) of the step's queries (-inf past the block); 16-byte loads
  alignas(16) float dsum[kStat][BT];   // -D = -(dO . O); 16-byte loads
  int2 blk[kStat];         // the step's query block (first query, count | full << 16)
  uint64_t kv_full, q_full[NH], q_empty[NH], stat_full[kStat], stat_empty[kStat], s_full[2], p_part[2], p_full[2], acc_done,
      drain;
  uint32_t tmem_base;
  int abort_flag;
};

template <int D, int NH, bool kHiLo>
__global__ void __launch_bounds__(384, 1)
    bwd_kv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                  const BwdParams p) {
  using Smem = KVSmem<D, NH>;
  static_assert(offsetof(Smem, lse2) % 16 == 0 && offsetof(Smem, dsum) % 16 == 0, "16-byte shared loads");
  extern __shared__ uint8_t smem_raw[];
  Smem& S = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  volatile int* abort_flag = &S.abort_flag;

  const int item = blockIdx.x;
  const int tile = __ldg(p.kt_order + item / p.Hkv);
  const int g = item % p.Hkv;                 // KV head
  const int G = p.group_size;                 // query heads per KV head
  const int k0 = __ldg(p.kt_k0 + tile);
  const int nk = __ldg(p.kt_nk + tile);
  const int qb_begin = __ldg(p.kt_qb_begin + tile);
  const int n_steps = (__ldg(p.kt_qb_begin + tile + 1) - qb_begin) * G;
  constexpr uint32_t cdV = 256, cdK = 256 + D;

  if (threadIdx.x == 0) {
    ptx::mbar_init(&S.kv_full, 1);
    for (int s = 0; s < NH; ++s) {
      ptx::mbar_init(&S.q_full[s], 1);
      ptx::mbar_init(&S.q_empty[s], 1);
    }
    for (int s = 0; s < kStat; ++s) {
      ptx::mbar_init(&S.stat_full[s], 1);
      ptx::mbar_init(&S.stat_empty[s], 8);   // one arrival per softmax warp
    }
    for (int h = 0; h < 2; ++h) {
      ptx::mbar_init(&S.s_full[h], 1);
      ptx::mbar_init(&S.p_part[h], 128);   // P^T, dS^T of the half's first 32 queries stored
      ptx::mbar_init(&S.p_full[h], 128);
    }
    ptx::mbar_init(&S.acc_done, 1);
    ptx::mbar_init(&S.drain, 1);
    S.abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(&S.tmem_base, 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = S.tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (ptx::elect_one()) {
      ptx::mbar_arrive_expect_tx(&S.kv_full, 2 * D * 256);
      for (int c = 0; c < D / 64; ++c) {
        ptx::tma_load_3d(S.k[c], &tm_k, &S.kv_full, c * 64, g, k0);
        ptx::tma_load_3d(S.v[c], &tm_v, &S.kv_full, c * 64, g, k0);
      }
      int issued = 0;
      for (int m = 0; m < 2 * n_steps; ++m) {   // half-steps: step m/2, queries (m%2)*64..
        const int n = m >> 1;
        const int st = m % NH;
        const uint32_t use = m / NH;
        const int qs = __ldg(&p.qb[qb_begin + n / G].x) + (m & 1) * kHalf;
        const int h = g * G + n % G;
        if (m >= NH && !ptx::mbar_wait(&S.q_empty[st], (use - 1) & 1, abort_flag, kWaitLimitNs)) break;
        ptx::mbar_arrive_expect_tx(&S.q_full[st], 2 * D * 128);
        for (int c = 0; c < D / 64; ++c) {
          ptx::tma_load_3d(S.q[st][c], &tm_q, &S.q_full[st], c * 64, h, qs);
          ptx::tma_load_3d(S.dO[st][c], &tm_do, &S.q_full[st], c * 64, h, qs);
        }
        issued = m + 1;
      }
      if (*abort_flag) {
        for (int m = (issued > NH ? issued - NH : 0); m < issued; ++m) ptx::mbar_drain(&S.q_full[m % NH], (m / NH) & 1);
        ptx::mbar_drain(&S.kv_full, 0);
      }
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ row terms
    // Loads kStat steps at a time (all their global loads in flight together)
    // and fetches the next batch's block entries ahead, so the ring stays
    // ahead of the softmax warpgroups.
    int2 pre[kStat];
#pragma unroll
    for (int x = 0; x < kStat; ++x) pre[x] = x < n_steps ? __ldg(&p.qb[qb_begin + x / G]) : make_int2(0, 0);
    bool ok = true;
    for (int n0 = 0; ok && n0 < n_steps; n0 += kStat) {
      int2 cur[kStat];
      float lv[kStat][BT / 32], dv[kStat][BT / 32];
#pragma unroll
      for (int x = 0; x < kStat; ++x) {
        cur[x] = pre[x];
        const int nn = n0 + kStat + x;
        pre[x] = nn < n_steps ? __ldg(&p.qb[qb_begin + nn / G]) : make_int2(0, 0);
      }
#pragma unroll
      for (int x = 0; x < kStat; ++x) {
        const int n = n0 + x;
        const int h = g * G + n % G;
        const int qs = cur[x].x, nq = cur[x].y & 0xFFFF;
        const float* lse_h = p.lse + static_cast<int64_t>(h) * p.F + qs;
        const float* dsum_h = p.dsum + static_cast<int64_t>(h) * p.F + qs;
#pragma unroll
        for (int y = 0; y < BT / 32; ++y) {
          const int c = lane + 32 * y;
          const bool in = n < n_steps && c < nq;
          lv[x][y] = in ? -__ldg(lse_h + c) * kLog2e : -INFINITY;
          dv[x][y] = in ? -__ldg(dsum_h + c) : 0.f;
        }
      }
#pragma unroll
      for (int x = 0; x < kStat; ++x) {
        const int n = n0 + x;
        if (n >= n_steps) break;
        const int st = n % kStat;
        const uint32_t use = n / kStat;
        ok = n < kStat || ptx::mbar_wait(&S.stat_empty[st], (use - 1) & 1, abort_flag, kWaitLimitNs);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
#pragma unroll
        for (int y = 0; y < BT / 32; ++y) {
          S.lse2[st][lane + 32 * y] = lv[x][y];
          S.dsum[st][lane + 32 * y] = dv[x][y];
        }
        if (lane == 0) S.blk[st] = cur[x];
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&S.stat_full[st]);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (ptx::elect_one()) {
      constexpr uint32_t idesc_s = ptx::idesc_bf16_f32(BT, kHalf, false, false);
      constexpr uint32_t idesc_acc = ptx::idesc_bf16_f32(BT, D, false, true);
      bool ok = ptx::mbar_wait(&S.kv_full, 0, abort_flag, kWaitLimitNs);
      ptx::tc_fence_after();
      const uint32_t k_base = ptx::smem_addr(S.k[0]);
      const uint32_t v_base = ptx::smem_addr(S.v[0]);
      // S^T, dP^T of one 64-query half-stage (K-major B operands, 64 rows)
      auto issue_sdp = [&](int m, int slot) {
        const uint32_t qb = ptx::smem_addr(S.q[m % NH][0]);
        const uint32_t ob = ptx::smem_addr(S.dO[m % NH][0]);
        const uint32_t cS = BT * slot, cdP = BT * slot + kHalf;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t aoff = (kk >> 2) * kBox + (kk & 3) * 32;
          const uint32_t boff = (kk >> 2) * kHalfBox + (kk & 3) * 32;
          ptx::mma_ss(tmem + cS, ptx::desc_add(ptx::sw128_desc(k_base, 16, 1024), aoff), ptx::desc_add(ptx::sw128_desc(qb, 16, 1024), boff),
                      idesc_s, kk > 0 ? 1u : 0u);
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t aoff = (kk >> 2) * kBox + (kk & 3) * 32;
          const uint32_t boff = (kk >> 2) * kHalfBox + (kk & 3) * 32;
          ptx::mma_ss(tmem + cdP, ptx::desc_add(ptx::sw128_desc(v_base, 16, 1024), aoff), ptx::desc_add(ptx::sw128_desc(ob, 16, 1024), boff),
                      idesc_s, kk > 0 ? 1u : 0u);
        }
        ptx::mma_commit(&S.s_full[slot]);
      };
      // dV += P^T dO_half, dK += dS^T Q_half (half-stages as MN-major B
      // operands: d-column groups one 64-row box apart; the precise mode adds
      // the low halves' products), then release the stage in two parts of 32
      // queries, each issued as soon as the softmax has stored that part's
      // P^T and dS^T (p_part, then p_full)
      auto issue_acc = [&](int m, int slot, bool first, uint32_t parity) {
        const uint32_t qb = ptx::smem_addr(S.q[m % NH][0]);
        const uint32_t ob = ptx::smem_addr(S.dO[m % NH][0]);
        const uint32_t cS = BT * slot, cdP = BT * slot + kHalf;
        for (int part = 0; part < 2; ++part) {
          if (!ptx::mbar_wait(part == 0 ? &S.p_part[slot] : &S.p_full[slot], parity, abort_flag, kWaitLimitNs))
            return false;
          ptx::tc_fence_after();
#pragma unroll
          for (int kk = part * (kHalf / 32); kk < (part + 1) * (kHalf / 32); ++kk) {
            const uint32_t acc = (first && kk == 0) ? 0u : 1u;
            const uint64_t bo = ptx::desc_add(ptx::sw128_desc(ob, kHalfBox, 1024), kk * 2048);
            const uint64_t bq = ptx::desc_add(ptx::sw128_desc(qb, kHalfBox, 1024), kk * 2048);
            ptx::mma_ts(tmem + cdV, tmem + cS + a_col(kk, false), bo, idesc_acc, acc);
            ptx::mma_ts(tmem + cdK, tmem + cdP + a_col(kk, false), bq, idesc_acc, acc);
            if constexpr (kHiLo) {
              ptx::mma_ts(tmem + cdV, tmem + cS + a_col(kk, true), bo, idesc_acc, 1u);
              ptx::mma_ts(tmem + cdK, tmem + cdP + a_col(kk, true), bq, idesc_acc, 1u);
            }
          }
        }
        ptx::mma_commit(&S.q_empty[m % NH]);
        return true;
      };
      auto wait_stage = [&](int m) {
        const bool r = ptx::mbar_wait(&S.q_full[m % NH], (m / NH) & 1, abort_flag, kWaitLimitNs);
        ptx::tc_fence_after();
        return r;
      };
      for (int n = 0; ok && n < n_steps; ++n) {
        if (!wait_stage(2 * n)) { ok = false; break; }
        issue_sdp(2 * n, 0);
        if (n > 0 && !issue_acc(2 * n - 1, 1, false, (n - 1) & 1)) { ok = false; break; }
        if (!wait_stage(2 * n + 1)) { ok = false; break; }
        issue_sdp(2 * n + 1, 1);
        if (!issue_acc(2 * n, 0, n == 0, n & 1)) { ok = false; break; }
      }
      if (ok && n_steps > 0) {
        const int last = n_steps - 1;
        if (issue_acc(2 * last + 1, 1, false, last & 1)) ptx::mma_commit(&S.acc_done);
      }
      ptx::mma_commit(&S.drain);
      ptx::mbar_drain(&S.drain, 0);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax
    const int half = (warp - 4) >> 2;        // which 64 queries of a step
    const int wq = warp & 3;
    const int t = wq * 32 + lane;
    const int j = k0 + t;                    // this thread's key
    const int se_j = t < nk ? __ldg(p.subtree_end + j) : -1;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem + lane_off + BT * half, tdP = tS + kHalf;
    const float sl2 = p.scale_log2;
    const uint64_t sl2x2 = ptx::f2(sl2, sl2);
    bool ok = true;
    for (int n = 0; n < n_steps; ++n) {
      const int sst = n % kStat;
      ok = ptx::mbar_wait(&S.stat_full[sst], (n / kStat) & 1, abort_flag, kWaitLimitNs) &&
           ptx::mbar_wait(&S.s_full[half], n & 1, abort_flag, kWaitLimitNs);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      ptx::tc_fence_after();
      const int2 blk = S.blk[sst];
      const int qs = blk.x, nq = blk.y & 0xFFFF;
      const bool full = (blk.y >> 16) & 1;
      // visible queries of this key form one column range [lo, hi) of the half:
      // i >= j (causal) and i < subtree_end[j], inside the block
      const int base = qs + half * kHalf;
      const int lo = full ? 0 : max(0, j - base);
      const int hi = full ? kHalf : min(min(nq - half * kHalf, kHalf), se_j - base);
      const float* l2s = S.lse2[sst] + half * kHalf;
      const float* dds = S.dsum[sst] + half * kHalf;
#pragma unroll
      for (int c = 0; c < kHalf / 32; ++c) {
        uint32_t us[32], ud[32];
        ptx::tmem_ld32(tS + c * 32, us);
        ptx::tmem_ld32(tdP + c * 32, ud);
        ptx::tmem_wait_ld();
        // exponent arguments s*scale*log2(e) - LSE*log2(e), two per instruction
        // (the row terms are stored negated, so a 16-byte load is two pairs)
        float arg[32];
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          const ulonglong2 nl = ptx::lds128u(l2s + c * 32 + e);
          ptx::unf2(ptx::fma2(ptx::f2(__uint_as_float(us[e]), __uint_as_float(us[e + 1])), sl2x2, nl.x), arg[e],
                    arg[e + 1]);
          ptx::unf2(ptx::fma2(ptx::f2(__uint_as_float(us[e + 2]), __uint_as_float(us[e + 3])), sl2x2, nl.y),
                    arg[e + 2], arg[e + 3]);
        }
        if (!full) {
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int col = c * 32 + e;
            arg[e] = (col >= lo && col < hi) ? arg[e] : -INFINITY;
          }
        }
        // P = 2^arg; dS = P * (dP - D), two per instruction
        uint32_t pp[16], pd[16];
        uint32_t pl[kHiLo ? 16 : 1], dl[kHiLo ? 16 : 1];
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          const ulonglong2 nd = ptx::lds128u(dds + c * 32 + e);
          const float p0 = ptx::ex2(arg[e]), p1 = ptx::ex2(arg[e + 1]);
          const float p2 = ptx::ex2(arg[e + 2]), p3 = ptx::ex2(arg[e + 3]);
          const uint64_t pa = ptx::f2(p0, p1), pb = ptx::f2(p2, p3);
          float d0, d1, d2, d3;
          ptx::unf2(ptx::mul2(pa, ptx::add2(ptx::f2(__uint_as_float(ud[e]), __uint_as_float(ud[e + 1])), nd.x)), d0, d1);
          ptx::unf2(ptx::mul2(pb, ptx::add2(ptx::f2(__uint_as_float(ud[e + 2]), __uint_as_float(ud[e + 3])), nd.y)), d2,
                    d3);
          if constexpr (kHiLo) {
            ptx::split_bf16x2(p0, p1, pp[e / 2], pl[e / 2]);
            ptx::split_bf16x2(p2, p3, pp[e / 2 + 1], pl[e / 2 + 1]);
            ptx::split_bf16x2(d0, d1, pd[e / 2], dl[e / 2]);
            ptx::split_bf16x2(d2, d3, pd[e / 2 + 1], dl[e / 2 + 1]);
          } else {
            pp[e / 2] = ptx::pack_bf16x2(p0, p1);
            pp[e / 2 + 1] = ptx::pack_bf16x2(p2, p3);
            pd[e / 2] = ptx::pack_bf16x2(d0, d1);
            pd[e / 2 + 1] = ptx::pack_bf16x2(d2, d3);
          }
        }
        // part c: columns 32c.. (already read above), high halves first
        ptx::tmem_st16(tS + c * 32, pp);
        ptx::tmem_st16(tdP + c * 32, pd);
        if constexpr (kHiLo) {
          ptx::tmem_st16(tS + c * 32 + 16, pl);
          ptx::tmem_st16(tdP + c * 32 + 16, dl);
        }
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        ptx::mbar_arrive(c == 0 ? &S.p_part[half] : &S.p_full[half]);
      }
      // the row terms of this step are no longer needed by this warp
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&S.stat_empty[sst]);
    }
    if (ok) {
      ok = ptx::mbar_wait(&S.acc_done, 0, abort_flag, kWaitLimitNs);
      ok = __all_sync(0xffffffffu, ok);
    }
    if (ok) {
      // epilogue: warpgroup of half 0 writes dV, the other dK
      ptx::tc_fence_after();
      const uint32_t col = half == 0 ? cdV : cdK;
      const float mul = half == 0 ? 1.f : p.scale;
      __nv_bfloat16* row = (half == 0 ? p.dv : p.dk) + (static_cast<int64_t>(j) * p.Hkv + g) * D;
      if (half == 1 && p.rope) {
        // dK w.r.t. the un-rotated keys: frequency chunk c pairs columns
        // 32c.. with 32c + D/2..
        const float pf = t < nk ? static_cast<float>(__ldg(p.depth + j)) : 0.f;
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
          uint32_t ua[32], ub[32];
          ptx::tmem_ld32(tmem + lane_off + col + c * 32, ua);
          ptx::tmem_ld32(tmem + lane_off + col + D / 2 + c * 32, ub);
          ptx::tmem_wait_ld();
          if (t < nk) store_rotated<32>(row, c * 32, D / 2, ua, ub, mul, pf, p);
        }
      } else {
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t u[32];
          ptx::tmem_ld32(tmem + lane_off + col + c * 32, u);
          ptx::tmem_wait_ld();
          if (t < nk) store_row32(row + c * 32, u, mul);
        }
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
  if (threadIdx.x == 0 && S.abort_flag && p.err) atomicExch(p.err, TPK_E_TIMEOUT);
}

// ----------------------------------------------------------------- pass 3
// Query-major dQ.  Each key block of the forward's list is split into two
// 64-key halves alternating between two TMEM slots (same ping-pong as pass 2):
//   MMA order per block i:  S/dP(i, half 0) | dQ(i-1, half 1) | S/dP(i, half 1) | dQ(i, half 0)
// K and V stream through an NH-deep ring of 64-key half-stages (64-row TMA
// boxes), each released as soon as its half's dQ product is issued.
// TMEM: slot h at [128h, 128h+128): S (64 cols) then dP (64 cols); dQ at
// [256, 256+D); the query tile's Q and dO (bf16, D/2 cols each) after it.
// dS (bf16) overwrites S of its slot in two 32-key parts (columns 32c..,
// high halves first, low halves 16 columns on in the precise mode), released
// to the dQ products one after the other (p_part, p_full).  Q and dO are the A
// operands of the S and dP products straight from TMEM, so shared memory only
// feeds the 64-key K / V halves: on this part an M=128, N=64 product took
// about 75 cycles with its A tile in shared memory and 32-42 with it in TMEM
// (the A tile read does not overlap the product).
// Warps: 0 TMA producer, 1 MMA issuer + TMEM owner, 4-7 softmax of half 0,
// 8-11 softmax of half 1 (thread t owns query row t).
template <int D, int NH>
struct QSmem {
  uint8_t q[D / 64][kBox];
  uint8_t dO[D / 64][kBox];
  uint8_t k[NH][D / 64][kHalfBox];
  uint8_t v[NH][D / 64][kHalfBox];
  uint64_t q_full, qt_full, kv_full[NH], kv_empty[NH], s_full[2], p_part[2], p_full[2], acc_done, drain;
  alignas(16) int se[2][2][kHalf];    // [half][buffer][key]: subtree_end of a masked block's keys (16-byte loads)
  uint64_t se_bar[2];        // per half: its warpgroup has staged se
  uint32_t tmem_base;
  int abort_flag;
};

template <int D, int NH, bool kHiLo>
__global__ void __launch_bounds__(384, 1)
    bwd_q_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                 const BwdParams p) {
  using Smem = QSmem<D, NH>;
  static_assert(offsetof(Smem, se) % 16 == 0, "16-byte shared loads of se");
  extern __shared__ uint8_t smem_raw[];
  Smem& S = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5;
  volatile int* abort_flag = &S.abort_flag;

  const int item = blockIdx.x;
  const int tile = __ldg(p.qt_order + item / p.Hq);
  const int h = item % p.Hq;
  const int kvh = h / p.group_size;
  const int q0 = __ldg(p.qt_q0 + tile);
  const int nq = __ldg(p.qt_nq + tile);
  const int kb_begin = __ldg(p.qt_kb_begin + tile);
  const int n_blocks = __ldg(p.qt_kb_begin + tile + 1) - kb_begin;
  constexpr uint32_t cdQ = 256;
  constexpr uint32_t cQt = 256 + D, cOt = 256 + D + D / 2;   // Q, dO (bf16 pairs)

  if (threadIdx.x == 0) {
    ptx::mbar_init(&S.q_full, 1);
    ptx::mbar_init(&S.qt_full, 256);   // every softmax thread, after its TMEM row copy
    for (int s = 0; s < NH; ++s) {
      ptx::mbar_init(&S.kv_full[s], 1);
      ptx::mbar_init(&S.kv_empty[s], 1);
    }
    for (int x = 0; x < 2; ++x) {
      ptx::mbar_init(&S.s_full[x], 1);
      ptx::mbar_init(&S.p_part[x], 128);   // dS of the half's first 32 keys stored
      ptx::mbar_init(&S.p_full[x], 128);
      ptx::mbar_init(&S.se_bar[x], 128);
    }
    ptx::mbar_init(&S.acc_done, 1);
    ptx::mbar_init(&S.drain, 1);
    S.abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(&S.tmem_base, 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = S.tmem_base;

  if (warp == 0) {
    if (ptx::elect_one()) {
      ptx::mbar_arrive_expect_tx(&S.q_full, 2 * D * 256);
      for (int c = 0; c < D / 64; ++c) {
        ptx::tma_load_3d(S.q[c], &tm_q, &S.q_full, c * 64, h, q0);
        ptx::tma_load_3d(S.dO[c], &tm_do, &S.q_full, c * 64, h, q0);
      }
      int issued = 0;
      for (int m = 0; m < 2 * n_blocks; ++m) {   // half-steps: block m/2, keys (m%2)*64..
        const int st = m % NH;
        const uint32_t use = m / NH;
        const int kb0 = __ldg(&p.kb[kb_begin + m / 2].x) + (m & 1) * kHalf;
        if (m >= NH && !ptx::mbar_wait(&S.kv_empty[st], (use - 1) & 1, abort_flag, kWaitLimitNs)) break;
        ptx::mbar_arrive_expect_tx(&S.kv_full[st], 2 * D * 128);
        for (int c = 0; c < D / 64; ++c) {
          ptx::tma_load_3d(S.k[st][c], &tm_k, &S.kv_full[st], c * 64, kvh, kb0);
          ptx::tma_load_3d(S.v[st][c], &tm_v, &S.kv_full[st], c * 64, kvh, kb0);
        }
        issued = m + 1;
      }
      if (*abort_flag) {
        for (int m = (issued > NH ? issued - NH : 0); m < issued; ++m) ptx::mbar_drain(&S.kv_full[m % NH], (m / NH) & 1);
        ptx::mbar_drain(&S.q_full, 0);
      }
    }
  } else if (warp == 1) {
    if (ptx::elect_one()) {
      constexpr uint32_t idesc_s = ptx::idesc_bf16_f32(BT, kHalf, false, false);
      constexpr uint32_t idesc_dq = ptx::idesc_bf16_f32(BT, D, false, true);
      bool ok = ptx::mbar_wait(&S.qt_full, 0, abort_flag, kWaitLimitNs);
      ptx::tc_fence_after();
      // S, dP of one 64-key half-stage (K-major B operands, 64 rows)
      auto issue_sdp = [&](int m, int slot) {
        const uint32_t kb = ptx::smem_addr(S.k[m % NH][0]);
        const uint32_t vb = ptx::smem_addr(S.v[m % NH][0]);
        const uint32_t cS = BT * slot, cdP = BT * slot + kHalf;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t boff = (kk >> 2) * kHalfBox + (kk & 3) * 32;
          ptx::mma_ts(tmem + cS, tmem + cQt + kk * 8, ptx::desc_add(ptx::sw128_desc(kb, 16, 1024), boff), idesc_s,
                      kk > 0 ? 1u : 0u);
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t boff = (kk >> 2) * kHalfBox + (kk & 3) * 32;
          ptx::mma_ts(tmem + cdP, tmem + cOt + kk * 8, ptx::desc_add(ptx::sw128_desc(vb, 16, 1024), boff), idesc_s,
                      kk > 0 ? 1u : 0u);
        }
        ptx::mma_commit(&S.s_full[slot]);
      };
      // dQ += dS K_half (half-stage as the MN-major B operand: d-column groups
      // one 64-row box apart, 16 keys = 2 KB per step); then release the stage
      // in two parts of 32 keys, each issued as soon as the softmax has
      // stored that part's dS (p_part, then p_full)
      auto issue_dq = [&](int m, int slot, bool first, uint32_t parity) {
        const uint32_t kb = ptx::smem_addr(S.k[m % NH][0]);
        const uint32_t cS = BT * slot;
        for (int part = 0; part < 2; ++part) {
          if (!ptx::mbar_wait(part == 0 ? &S.p_part[slot] : &S.p_full[slot], parity, abort_flag, kWaitLimitNs))
            return false;
          ptx::tc_fence_after();
#pragma unroll
          for (int kk = part * (kHalf / 32); kk < (part + 1) * (kHalf / 32); ++kk) {
            const uint64_t bk = ptx::desc_add(ptx::sw128_desc(kb, kHalfBox, 1024), kk * 2048);
            ptx::mma_ts(tmem + cdQ, tmem + cS + a_col(kk, false), bk, idesc_dq, (first && kk == 0) ? 0u : 1u);
            if constexpr (kHiLo) ptx::mma_ts(tmem + cdQ, tmem + cS + a_col(kk, true), bk, idesc_dq, 1u);
          }
        }
        ptx::mma_commit(&S.kv_empty[m % NH]);
        return true;
      };
      auto wait_stage = [&](int m) {
        const bool r = ptx::mbar_wait(&S.kv_full[m % NH], (m / NH) & 1, abort_flag, kWaitLimitNs);
        ptx::tc_fence_after();
        return r;
      };
      for (int i = 0; ok && i < n_blocks; ++i) {
        if (!wait_stage(2 * i)) { ok = false; break; }
        issue_sdp(2 * i, 0);
        if (i > 0 && !issue_dq(2 * i - 1, 1, false, (i - 1) & 1)) { ok = false; break; }
        if (!wait_stage(2 * i + 1)) { ok = false; break; }
        issue_sdp(2 * i + 1, 1);
        if (!issue_dq(2 * i, 0, i == 0, i & 1)) { ok = false; break; }
      }
      if (ok && n_blocks > 0) {
        const int last = n_blocks - 1;
        if (issue_dq(2 * last + 1, 1, false, last & 1)) ptx::mma_commit(&S.acc_done);
      }
      ptx::mma_commit(&S.drain);
      ptx::mbar_drain(&S.drain, 0);
    }
  } else if (warp >= 4) {
    const int half = (warp - 4) >> 2;        // which 64 keys of a block
    const int wq = warp & 3;
    const int t = wq * 32 + (threadIdx.x & 31);
    const int i = q0 + t;                    // this thread's query
    const bool row_ok = t < nq;
    const float l2 = row_ok ? __ldg(p.lse + static_cast<int64_t>(h) * p.F + i) * kLog2e : 0.f;
    const float dd = row_ok ? __ldg(p.dsum + static_cast<int64_t>(h) * p.F + i) : 0.f;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem + lane_off + BT * half, tdP = tS + kHalf;
    const float sl2 = p.scale_log2;
    const uint64_t sl2x2 = ptx::f2(sl2, sl2), nl2x2 = ptx::f2(-l2, -l2), ndd2 = ptx::f2(-dd, -dd);
    // row t of the query tile into TMEM lane t: warpgroup 0 copies Q, 1 copies
    // dO.  The tile sits in shared memory as 128-byte-swizzled boxes of 64
    // elements (16-byte chunk c of row t at chunk c ^ (t % 8)); TMEM column w
    // holds elements 2w, 2w+1.
    bool ok = ptx::mbar_wait(&S.q_full, 0, abort_flag, kWaitLimitNs);
    ok = __all_sync(0xffffffffu, ok);
    if (ok) {
      const uint8_t* box0 = half == 0 ? S.q[0] : S.dO[0];
      const uint32_t dst = tmem + lane_off + (half == 0 ? cQt : cOt);
#pragma unroll
      for (int b = 0; b < D / 64; ++b) {
        uint32_t w[32];
        const uint8_t* row = box0 + b * kBox + t * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 v = *reinterpret_cast<const uint4*>(row + ((c ^ (t & 7)) << 4));
          w[4 * c] = v.x;
          w[4 * c + 1] = v.y;
          w[4 * c + 2] = v.z;
          w[4 * c + 3] = v.w;
        }
        ptx::tmem_st32(dst + b * 32, w);
      }
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      ptx::mbar_arrive(&S.qt_full);
    }
    int2 next = n_blocks > 0 ? __ldg(&p.kb[kb_begin]) : make_int2(0, 0);
    int n_masked = 0;   // masked blocks so far (selects the subtree_end buffer)
    for (int b = 0; ok && b < n_blocks; ++b) {
      const int2 blk = next;   // fetched one block ahead
      if (b + 1 < n_blocks) next = __ldg(&p.kb[kb_begin + b + 1]);
      ok = ptx::mbar_wait(&S.s_full[half], b & 1, abort_flag, kWaitLimitNs);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      ptx::tc_fence_after();
      const int kb0 = blk.x, nkb = blk.y & 0xFFFF;
      const bool full = (blk.y >> 16) & 1;
      const int base = kb0 + half * kHalf;     // first key of this half
      const int* se = S.se[half][n_masked & 1];
      if (!full) {
        // key j = base + col is visible to query i iff j <= i < subtree_end[j]:
        // the warpgroup stages the half's subtree_end in shared memory (one
        // load per thread; 0 past the block's end, which hides the column)
        // and meets at its se_bar (bounded wait); two buffers by the parity of
        // the masked-block count, as in the forward
        if (t < kHalf) S.se[half][n_masked & 1][t] = half * kHalf + t < nkb ? __ldg(p.subtree_end + base + t) : 0;
        ptx::mbar_arrive(&S.se_bar[half]);
        ok = ptx::mbar_wait(&S.se_bar[half], n_masked & 1, abort_flag, kWaitLimitNs);
        ok = __all_sync(0xffffffffu, ok);
        ++n_masked;
        if (!ok) break;
      }
      const int cmax = i - base;               // columns <= cmax hold keys j <= i
#pragma unroll
      for (int c = 0; c < kHalf / 32; ++c) {
        uint32_t us[32], ud[32];
        ptx::tmem_ld32(tS + c * 32, us);
        ptx::tmem_ld32(tdP + c * 32, ud);
        ptx::tmem_wait_ld();
        float arg[32];
#pragma unroll
        for (int e = 0; e < 32; e += 2)
          ptx::unf2(ptx::fma2(ptx::f2(__uint_as_float(us[e]), __uint_as_float(us[e + 1])), sl2x2, nl2x2), arg[e],
                    arg[e + 1]);
        if (!full) {
#pragma unroll
          for (int e = 0; e < 32; e += 4) {
            const int4 v = ptx::lds128i(se + c * 32 + e);
            const int cc = c * 32 + e;
            if (!(row_ok && cc <= cmax && i < v.x)) arg[e] = -INFINITY;
            if (!(row_ok && cc + 1 <= cmax && i < v.y)) arg[e + 1] = -INFINITY;
            if (!(row_ok && cc + 2 <= cmax && i < v.z)) arg[e + 2] = -INFINITY;
            if (!(row_ok && cc + 3 <= cmax && i < v.w)) arg[e + 3] = -INFINITY;
          }
        } else if (!row_ok) {
#pragma unroll
          for (int e = 0; e < 32; ++e) arg[e] = -INFINITY;
        }
        uint32_t pd[16];
        uint32_t dl[kHiLo ? 16 : 1];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const uint64_t pp = ptx::f2(ptx::ex2(arg[e]), ptx::ex2(arg[e + 1]));
          float d0, d1;
          ptx::unf2(ptx::mul2(pp, ptx::add2(ptx::f2(__uint_as_float(ud[e]), __uint_as_float(ud[e + 1])), ndd2)), d0, d1);
          if constexpr (kHiLo)
            ptx::split_bf16x2(d0, d1, pd[e / 2], dl[e / 2]);
          else
            pd[e / 2] = ptx::pack_bf16x2(d0, d1);
        }
        // part c: columns 32c.. (already read above), high halves first
        ptx::tmem_st16(tS + c * 32, pd);
        if constexpr (kHiLo) ptx::tmem_st16(tS + c * 32 + 16, dl);
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        ptx::mbar_arrive(c == 0 ? &S.p_part[half] : &S.p_full[half]);
      }
    }
    if (ok) {
      ok = ptx::mbar_wait(&S.acc_done, 0, abort_flag, kWaitLimitNs);
      ok = __all_sync(0xffffffffu, ok);
    }
    if (ok) {
      ptx::tc_fence_after();
      __nv_bfloat16* row = p.dq + (static_cast<int64_t>(i) * p.Hq + h) * D;
      if (p.rope) {
        // dQ w.r.t. the un-rotated queries: each warpgroup takes a quarter of
        // the columns, frequencies [half*D/4, +D/4), and their partners D/2 on
        constexpr int W = D / 4;
        const int f0 = half * W;
        const float pf = row_ok ? static_cast<float>(__ldg(p.depth + i)) : 0.f;
        uint32_t ua[W], ub[W];
        if constexpr (W == 32) {
          ptx::tmem_ld32(tmem + lane_off + cdQ + f0, ua);
          ptx::tmem_ld32(tmem + lane_off + cdQ + D / 2 + f0, ub);
        } else {
          ptx::tmem_ld16(tmem + lane_off + cdQ + f0, ua);
          ptx::tmem_ld16(tmem + lane_off + cdQ + D / 2 + f0, ub);
        }
        ptx::tmem_wait_ld();
        if (row_ok) store_rotated<W>(row, f0, D / 2, ua, ub, p.scale, pf, p);
      } else {
        // each warpgroup writes half of the head dimension
#pragma unroll
        for (int c = half * (D / 64); c < (half + 1) * (D / 64); ++c) {
          uint32_t u[32];
          ptx::tmem_ld32(tmem + lane_off + cdQ + c * 32, u);
          ptx::tmem_wait_ld();
          if (row_ok) store_row32(row + c * 32, u, p.scale);
        }
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
  if (threadIdx.x == 0 && S.abort_flag && p.err) atomicExch(p.err, TPK_E_TIMEOUT);
}

template <int D, int NH, bool kHiLo>
int launch_kv(const BwdParams& prm, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
              const CUtensorMap& tdo, int64_t n_ktiles, cudaStream_t stream) {
  constexpr size_t smem = sizeof(KVSmem<D, NH>) + 1024;
  static_assert(smem <= 227 * 1024, "shared memory");
  static PerContext<int> cfg;   // the shared-memory limit is per context (per device)
  int st = set_smem_once(cfg, bwd_kv_kernel<D, NH, kHiLo>, smem);
  if (st != TPK_OK) return st;
  const int64_t items = n_ktiles * prm.Hkv;
  if (items > 0x7fffffff) return TPK_E_OVERFLOW;
  if (items > 0)
    bwd_kv_kernel<D, NH, kHiLo><<<static_cast<unsigned>(items), 384, smem, stream>>>(tq, tk, tv, tdo, prm);
  return cuda_status(cudaGetLastError());
}

template <int D, int NH, bool kHiLo>
int launch_q(const BwdParams& prm, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
             const CUtensorMap& tdo, int64_t n_qtiles, cudaStream_t stream) {
  constexpr size_t smem = sizeof(QSmem<D, NH>) + 1024;
  static_assert(smem <= 227 * 1024, "shared memory");
  static PerContext<int> cfg;
  int st = set_smem_once(cfg, bwd_q_kernel<D, NH, kHiLo>, smem);
  if (st != TPK_OK) return st;
  const int64_t items = n_qtiles * prm.Hq;
  if (items > 0x7fffffff) return TPK_E_OVERFLOW;
  if (items > 0)
    bwd_q_kernel<D, NH, kHiLo><<<static_cast<unsigned>(items), 384, smem, stream>>>(tq, tk, tv, tdo, prm);
  return cuda_status(cudaGetLastError());
}

// One phase of the backward, options already checked.
int bwd_phase(int32_t phase, const Plan& P, const void* dev_image, const void* q, const void* k, const void* v,
              const void* o, const float* lse, const void* dout, void* dq, void* dk, void* dv, int32_t Hq,
              int32_t Hkv, int32_t d, float scale, bool precise, double rope_base, const void* o_lo,
              void* workspace, int32_t* dev_err, cudaStream_t s) {
  int st;
  if (phase == TPK_BWD_PREP) {
    const int64_t rows_per_block = 8 * (32 / (d / 8));   // 8 warps, 32/(d/8) rows each
    int64_t blocks = (P.F * Hq + rows_per_block - 1) / rows_per_block;
    const int64_t cap = int64_t{num_sms()} * 32;
    if (blocks > cap) blocks = cap;
    bwd_prep_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(
        static_cast<const __nv_bfloat16*>(o), precise ? static_cast<const __nv_bfloat16*>(o_lo) : nullptr,
        static_cast<const __nv_bfloat16*>(dout), static_cast<float*>(workspace), P.F, Hq, d);
    return cuda_status(cudaGetLastError());
  }
  CUtensorMap tq, tk, tv, tdo;
  if ((st = make_map_bf16(&tq, q, P.F, Hq, d, 128)) != TPK_OK) return st;
  if ((st = make_map_bf16(&tk, k, P.F, Hkv, d, 128)) != TPK_OK) return st;
  if ((st = make_map_bf16(&tv, v, P.F, Hkv, d, 128)) != TPK_OK) return st;
  if ((st = make_map_bf16(&tdo, dout, P.F, Hq, d, 128)) != TPK_OK) return st;
  const uint8_t* img = static_cast<const uint8_t*>(dev_image);
  BwdParams prm;
  prm.qt_q0 = reinterpret_cast<const int32_t*>(img + P.off_qt_q0);
  prm.qt_nq = reinterpret_cast<const int32_t*>(img + P.off_qt_nq);
  prm.qt_kb_begin = reinterpret_cast<const int32_t*>(img + P.off_qt_kb_begin);
  prm.kb = reinterpret_cast<const int2*>(img + P.off_kb);
  prm.qt_order = reinterpret_cast<const int32_t*>(img + P.off_qt_order);
  prm.kt_k0 = reinterpret_cast<const int32_t*>(img + P.off_kt_k0);
  prm.kt_nk = reinterpret_cast<const int32_t*>(img + P.off_kt_nk);
  prm.kt_qb_begin = reinterpret_cast<const int32_t*>(img + P.off_kt_qb_begin);
  prm.qb = reinterpret_cast<const int2*>(img + P.off_qb);
  prm.kt_order = reinterpret_cast<const int32_t*>(img + P.off_kt_order);
  prm.subtree_end = reinterpret_cast<const int32_t*>(img + P.off_subtree_end);
  prm.lse = lse;
  prm.dsum = static_cast<float*>(workspace);
  prm.dq = static_cast<__nv_bfloat16*>(dq);
  prm.dk = static_cast<__nv_bfloat16*>(dk);
  prm.dv = static_cast<__nv_bfloat16*>(dv);
  prm.F = static_cast<int32_t>(P.F);
  prm.Hq = Hq;
  prm.Hkv = Hkv;
  prm.group_size = Hq / Hkv;
  prm.scale = scale;
  prm.scale_log2 = scale * kLog2e;
  prm.err = dev_err;
  prm.depth = reinterpret_cast<const int32_t*>(img + P.off_depth);
  prm.rope = rope_base > 0.0 ? 1 : 0;
  for (int i = 0; i < 64; ++i) {
    // turns per unit depth of frequency i: base^(-2i/d) / (2 pi), as hi + lo
    const double t = i < d / 2 && prm.rope ? std::pow(rope_base, -2.0 * i / d) / 6.283185307179586476925286766559 : 0.0;
    prm.rope_hi[i] = static_cast<float>(t);
    prm.rope_lo[i] = static_cast<float>(t - static_cast<double>(prm.rope_hi[i]));
  }
  const int64_t nkt = static_cast<int64_t>(P.kt_k0.size()), nqt = static_cast<int64_t>(P.qt_q0.size());
  if (phase == TPK_BWD_DKDV) {
    // the dK/dV pass streams Q and dO in 64-query half-stages
    CUtensorMap tq64, tdo64;
    if ((st = make_map_bf16(&tq64, q, P.F, Hq, d, 64)) != TPK_OK) return st;
    if ((st = make_map_bf16(&tdo64, dout, P.F, Hq, d, 64)) != TPK_OK) return st;
    if (d == 128)
      return precise ? launch_kv<128, 4, true>(prm, tq64, tk, tv, tdo64, nkt, s)
                     : launch_kv<128, 4, false>(prm, tq64, tk, tv, tdo64, nkt, s);
    return precise ? launch_kv<64, 8, true>(prm, tq64, tk, tv, tdo64, nkt, s)
                   : launch_kv<64, 8, false>(prm, tq64, tk, tv, tdo64, nkt, s);
  }
  // the dQ pass streams K and V in 64-key half-stages
  CUtensorMap tk64, tv64;
  if ((st = make_map_bf16(&tk64, k, P.F, Hkv, d, 64)) != TPK_OK) return st;
  if ((st = make_map_bf16(&tv64, v, P.F, Hkv, d, 64)) != TPK_OK) return st;
  if (d == 128)
    return precise ? launch_q<128, 4, true>(prm, tq, tk64, tv64, tdo, nqt, s)
                   : launch_q<128, 4, false>(prm, tq, tk64, tv64, tdo, nqt, s);
  return precise ? launch_q<64, 8, true>(prm, tq, tk64, tv64, tdo, nqt, s)
                 : launch_q<64, 8, false>(prm, tq, tk64, tv64, tdo, nqt, s);
}

}  // namespace
}  // namespace tpk

extern "C" size_t tpk_attn_workspace_bytes(const tpk_plan* plan, int32_t Hq, int32_t Hkv, int32_t d, int32_t backward) {
  (void)Hkv;
  (void)d;
  if (!plan || !backward || Hq <= 0) return 0;
  // D[h, f] = dO . O, fp32 [Hq, F]
  return (static_cast<size_t>(Hq) * static_cast<size_t>(plan->p.F) * 4 + 255) & ~size_t(255);
}

extern "C" int tpk_tree_attn_bwd_ex(int32_t phase, const tpk_plan* plan, const void* dev_image, const void* q,
                                    const void* k, const void* v, const void* o, const float* lse, const void* dout,
                                    void* dq, void* dk, void* dv, int32_t Hq, int32_t Hkv, int32_t d, float scale,
                                    const tpk_attn_opts* opts, void* workspace, size_t ws_bytes, int32_t* dev_err,
                                    void* stream) {
  using namespace tpk;
  if (!plan || phase < TPK_BWD_ALL || phase > TPK_BWD_DQ) return TPK_E_ARG;
  if (Hq <= 0 || Hkv <= 0 || !(scale > 0.f)) return TPK_E_ARG;
  if ((d != 64 && d != 128) || Hq % Hkv != 0) return TPK_E_UNSUPPORTED;
  const bool all = phase == TPK_BWD_ALL;
  const bool prep = all || phase == TPK_BWD_PREP, kv = all || phase == TPK_BWD_DKDV, qp = all || phase == TPK_BWD_DQ;
  if (prep && (!o || !dout)) return TPK_E_ARG;
  if ((kv || qp) && (!dev_image || !q || !k || !v || !lse || !dout)) return TPK_E_ARG;
  if ((kv && (!dk || !dv)) || (qp && !dq)) return TPK_E_ARG;
  const bool precise = opts && opts->precision == TPK_PREC_PRECISE;
  const double rope_base = opts ? opts->rope_base : 0.0;
  const void* o_lo = opts ? opts->o_lo : nullptr;
  if (opts && opts->precision != TPK_PREC_FAST && opts->precision != TPK_PREC_PRECISE) return TPK_E_ARG;
  if (!(rope_base == 0.0 || rope_base > 1.0)) return TPK_E_ARG;
  if ((reinterpret_cast<uintptr_t>(dq) | reinterpret_cast<uintptr_t>(dk) | reinterpret_cast<uintptr_t>(dv) |
       reinterpret_cast<uintptr_t>(o) | reinterpret_cast<uintptr_t>(dout) | reinterpret_cast<uintptr_t>(o_lo)) % 16)
    return TPK_E_ARG;
  const Plan& P = plan->p;
  // the fused inverse rotation forms the angle from the depth in fp32
  if (rope_base > 1.0 && P.max_depth >= (int64_t{1} << 24)) return TPK_E_UNSUPPORTED;
  if (P.F == 0) return TPK_OK;
  const size_t need = tpk_attn_workspace_bytes(plan, Hq, Hkv, d, 1);
  if (!workspace || ws_bytes < need || reinterpret_cast<uintptr_t>(workspace) % 256) return TPK_E_WORKSPACE;
  int st = check_device();
  if (st != TPK_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  for (int32_t ph = TPK_BWD_PREP; ph <= TPK_BWD_DQ; ++ph) {
    if (!all && ph != phase) continue;
    st = bwd_phase(ph, P, dev_image, q, k, v, o, lse, dout, dq, dk, dv, Hq, Hkv, d, scale, precise, rope_base, o_lo,
                   workspace, dev_err, s);
    if (st != TPK_OK) return st;
  }
  return TPK_OK;
}

extern "C" int tpk_tree_attn_bwd_phase(int32_t phase, const tpk_plan* plan, const void* dev_image, const void* q,
                                       const void* k, const void* v, const void* o, const float* lse,
                                       const void* dout, void* dq, void* dk, void* dv, int32_t Hq, int32_t Hkv,
                                       int32_t d, float scale, void* workspace, size_t ws_bytes, int32_t* dev_err,
                                       void* stream) {
  if (phase < TPK_BWD_PREP || phase > TPK_BWD_DQ) return TPK_E_ARG;
  return tpk_tree_attn_bwd_ex(phase, plan, dev_image, q, k, v, o, lse, dout, dq, dk, dv, Hq, Hkv, d, scale, nullptr,
                              workspace, ws_bytes, dev_err, stream);
}

extern "C" int tpk_tree_attn_bwd(const tpk_plan* plan, const void* dev_image, const void* q, const void* k,
                                 const void* v, const void* o, const float* lse, const void* dout, void* dq, void* dk,
                                 void* dv, int32_t Hq, int32_t Hkv, int32_t d, float scale, void* workspace,
                                 size_t ws_bytes, int32_t* dev_err, void* stream) {
  if (!plan || !dev_image || !q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv) return TPK_E_ARG;
  return tpk_tree_attn_bwd_ex(TPK_BWD_ALL, plan, dev_image, q, k, v, o, lse, dout, dq, dk, dv, Hq, Hkv, d, scale,
                              nullptr, workspace, ws_bytes, dev_err, stream);
}

// ---------------------------------------------------------------------------
// Backward without any device allocation by the caller.
//
// Some callers cannot hand the library a workspace: hosts that own all device
// memory and give their plugins none at call time, code that must not call
// cudaMalloc/cudaFree because those calls can synchronise the device, and C
// runtimes with no device allocator at all.  For them the backward's only
// scratch -- the fp32 row terms D[h, f] = dO . O -- lives in this fixed,
// file-scope device array instead.  Every GPU that loads the library keeps it
// (32 MiB) until the process exits.
// ---------------------------------------------------------------------------
namespace tpk {
namespace {

constexpr size_t kStaticScratchBytes = size_t{32} << 20;   // 32 MiB: Hq * F <= 8,388,608
static __device__ __align__(256) uint8_t g_bwd_scratch[kStaticScratchBytes];

// Device address of g_bwd_scratch in the current context, looked up once per
// context (with it current) and cached by the context's unique id: another
// device, a context the caller made current, or the context that replaces one
// destroyed by cudaDeviceReset each get their own lookup, never a stale
// address.  In host code the name g_bwd_scratch is a host-side stand-in, not
// a device address, so kernels only ever receive the looked-up pointer.
PerContext<void*> g_scratch_addr;

int scratch_address(void** out) {
  return g_scratch_addr.get(out, [](void** p) {
    *p = nullptr;
    return (cudaGetSymbolAddress(p, g_bwd_scratch) == cudaSuccess && *p) ? TPK_OK : TPK_E_CUDA;
  });
}

}  // namespace
}  // namespace tpk

extern "C" int tpk_tree_attn_bwd_noalloc(const tpk_plan* plan, const void* dev_image, const void* q, const void* k,
                                         const void* v, const void* o, const float* lse, const void* dout, void* dq,
                                         void* dk, void* dv, int32_t Hq, int32_t Hkv, int32_t d, float scale,
                                         int32_t* dev_err, void* stream) {
  using namespace tpk;
  if (!plan || Hq <= 0 || Hkv <= 0) return TPK_E_ARG;
  const size_t need = tpk_attn_workspace_bytes(plan, Hq, Hkv, d, 1);
  if (need > kStaticScratchBytes) return TPK_E_SCRATCH_LIMIT;
  void* scratch = nullptr;
  int st = scratch_address(&scratch);
  if (st != TPK_OK) return st;
  // D is written in full by the first phase before anything reads it, so the
  // shared array needs no clearing between calls.
  return tpk_tree_attn_bwd(plan, dev_image, q, k, v, o, lse, dout, dq, dk, dv, Hq, Hkv, d, scale, scratch,
                           kStaticScratchBytes, dev_err, stream);
}
