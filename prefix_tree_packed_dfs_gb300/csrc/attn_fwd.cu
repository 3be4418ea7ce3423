// Tree attention forward on tcgen05 (sm_103a).
//
// What it computes ("Prefix Tree Packing in ART", section "Token-mixing
// layers"; "DAG packing", section "The mask"): for every forwarded query f and
// query head h, softmax attention over the keys visible to f -- f itself and
// its ancestors, i.e. keys j with j <= f < subtree_end[j] (the [enter, exit]
// interval test) -- and the natural-log LSE.
//
// Work decomposition.  Queries are cut into 128-row tiles on a per-row grid.
// The keys any query of tile [q0, q1) can see are the ancestors of q0 plus the
// tile itself (an ancestor of a later query that precedes q0 contains q0 in
// its subtree).  The planner lists them as key blocks of <= 128 keys taken
// from the merged ancestor intervals, flagging blocks visible to the whole
// tile ("full", no mask) -- the "one fully visible block per ancestor segment
// plus a causal triangle" of the pages.  Blocks off the ancestor chain are
// never visited, so work follows forwarded tokens, not raw ones.
//
// One CTA = one (query tile, pair of query heads sharing a KV head).  Both
// heads use the same K/V blocks, loaded once.  Warp roles:
//   warp 0      TMA producer: Q tiles once, then K and V blocks of 128 keys
//               through an NS-stage ring (separate full/empty barriers)
//   warp 1      MMA issuer (one thread) and TMEM owner
//   warps 4..   one softmax warpgroup per head slot; thread t owns query row t
// TMEM (512 columns): S_s at [128s, 128s+128) fp32 and O_s at [256 + D*s, +D)
// fp32, which fills it: QK^T reads Q from shared memory.  P_s (bf16) is
// written over the first 64 columns of S_s and fed to the PV product straight
// from TMEM, in two parts of half the keys: the softmax releases the first
// part (p_half) before computing the second (p_full), so the first part's PV
// products run meanwhile.  The MMA thread interleaves the two head slots
// (PV_0(i-1), S_0(i), PV_1(i-1), S_1(i)) so one slot's softmax overlaps the
// other slot's matrix products.
// With a GQA group of one (or an odd size) a CTA takes a single head and its
// two slots take the two 64-key halves of every block instead (split over
// keys inside the CTA): each slot keeps its own O, running maximum and row
// sum, merged once at the end.  S_s then needs 64 columns, which leaves room
// for the Q tile in TMEM ([128 + 2D, +D/2), copied there by the softmax warps
// once), so QK^T takes its A operand from TMEM -- measured 1.06-1.15x faster
// than whole blocks per slot with Q in shared memory.  With two heads the
// same 64-key form measured 1.16-1.24x slower than the layout above: its
// shorter products no longer cover the softmax of the other slot.
// Online softmax with a lazily raised running maximum: O and the row sum are
// rescaled only when the block maximum exceeds the one in use by more than
// 2^8, which keeps exponentials <= 256 and skips almost every rescale.
// P is stored part by part: part c (half of the S columns' keys) at column
// c*kCols/2, as bf16.  The precise mode stores the bf16 rounding of what that
// leaves out kCols/4 columns further and adds its PV product, so P enters PV
// with about 16 significant bits; it can also write the bf16 rounding
// residual of O next to O, for a backward that forms dO . O before O's
// rounding.
#include <cuda_bf16.h>

#include "common.cuh"
#include "plan_handle.h"
#include "ptx.cuh"

namespace tpk {
namespace {

constexpr int BM = 128;          // query rows per tile
constexpr int kBlock = 128;      // keys per block (one K/V stage)
constexpr int kBox = BM * 128;   // bytes of one 128-row x 64-element swizzled box
constexpr float kRescaleThreshold = 8.0f;   // log2 units
// Register split (384 threads): the producer / MMA
// warpgroup gives registers up to the two softmax warpgroups, which hold a
// 64-column score row per thread.
constexpr uint32_t kRegsCtl = 56;
constexpr uint32_t kRegsSoftmax = 216;
constexpr int kRegsNeeded = 128 * kRegsCtl + 256 * kRegsSoftmax;

struct FwdParams {
  const int32_t* qt_q0;
  const int32_t* qt_nq;
  const int32_t* qt_kb_begin;
  const int2* kb;
  const int32_t* qt_order;
  const int32_t* subtree_end;
  __nv_bfloat16* o;
  __nv_bfloat16* o_lo;   // precise mode: O - bf16(O), or null
  float* lse;
  int32_t F, Hq, n_hgroups, group_size;
  float scale_log2;
  int32_t* err;
};

template <int D, int HPC, int NS>
struct FwdSmem {
  uint8_t q[HPC][D / 64][kBox];
  uint8_t k[NS][D / 64][kBox];
  uint8_t v[NS][D / 64][kBox];
  uint64_t q_full, qt_full;
  uint64_t k_full[NS], v_full[NS], k_empty[NS], v_empty[NS];
  uint64_t s_full[2], p_half[2], p_full[2], o_done[2];
  uint64_t mrg_bar;          // single-head CTAs: the two slots swap (max, sum) per row
  float mrg[2][2][BM];       // [slot][max, sum][row]
  alignas(16) int se[2][2][kBlock];   // [slot][buffer][key]: subtree_end of a masked block's keys (16-byte loads)
  uint64_t se_bar[2];        // per slot: its warpgroup has staged se
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};

template <int D, int HPC, int NS>
constexpr size_t fwd_smem_bytes() {
  return sizeof(FwdSmem<D, HPC, NS>) + 1024;
}

template <int D, int HPC, int NS, bool kHiLo>
__global__ void __launch_bounds__(384, 1)
    tree_attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
  using Smem = FwdSmem<D, HPC, NS>;
  static_assert(offsetof(Smem, se) % 16 == 0, "16-byte shared loads of se");
  extern __shared__ uint8_t smem_raw[];
  Smem& S = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5;
  volatile int* abort_flag = &S.abort_flag;
  constexpr bool kSplit = HPC == 1;
  // keys per S accumulator: a whole block (two heads) or one half (one head)
  constexpr int kCols = kSplit ? kBlock / 2 : kBlock;
  // TMEM columns: S_s at kCols*s (fp32), O_s at cO0 + D*s (fp32), and with
  // one head its Q tile at cQ0 (bf16 pairs)
  constexpr uint32_t cO0 = 2 * kCols, cQ0 = 2 * kCols + 2 * D;
  static_assert(cQ0 + (kSplit ? D / 2 : 0) <= 512, "TMEM columns");

  const int item = blockIdx.x;
  const int tile = __ldg(p.qt_order + item / p.n_hgroups);
  const int h0 = (item % p.n_hgroups) * HPC;
  const int kvh = h0 / p.group_size;
  const int q0 = __ldg(p.qt_q0 + tile);
  const int nq = __ldg(p.qt_nq + tile);
  const int kb_begin = __ldg(p.qt_kb_begin + tile);
  const int n_blocks = __ldg(p.qt_kb_begin + tile + 1) - kb_begin;

  if (threadIdx.x == 0) {
    ptx::mbar_init(&S.q_full, 1);
    ptx::mbar_init(&S.qt_full, 256);   // one head: every softmax thread, after its rows of Q are in TMEM
    for (int s = 0; s < NS; ++s) {
      ptx::mbar_init(&S.k_full[s], 1);
      ptx::mbar_init(&S.v_full[s], 1);
      ptx::mbar_init(&S.k_empty[s], 1);
      ptx::mbar_init(&S.v_empty[s], 1);
    }
    ptx::mbar_init(&S.mrg_bar, 256);
    for (int h = 0; h < 2; ++h) {
      ptx::mbar_init(&S.se_bar[h], 128);
      ptx::mbar_init(&S.s_full[h], 1);
      ptx::mbar_init(&S.p_half[h], 128);   // P of the first half of the S columns stored
      ptx::mbar_init(&S.p_full[h], 128);
      ptx::mbar_init(&S.o_done[h], 1);
    }
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

  if (warp < 4) {
  ptx::regs_dec<kRegsCtl>();
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (ptx::elect_one()) {
      ptx::prefetch_tensormap(&tm_q);
      ptx::prefetch_tensormap(&tm_k);
      ptx::prefetch_tensormap(&tm_v);
      ptx::mbar_arrive_expect_tx(&S.q_full, HPC * D * 256);
      for (int s = 0; s < HPC; ++s)
        for (int c = 0; c < D / 64; ++c) ptx::tma_load_3d(S.q[s][c], &tm_q, &S.q_full, c * 64, h0 + s, q0);
      int issued = 0;
      for (int i = 0; i < n_blocks; ++i) {
        const int st = i % NS;
        const uint32_t use = i / NS;
        const int k0 = __ldg(&p.kb[kb_begin + i].x);
        if (i >= NS && !ptx::mbar_wait(&S.k_empty[st], (use - 1) & 1, abort_flag, kWaitLimitNs)) break;
        ptx::mbar_arrive_expect_tx(&S.k_full[st], D * 256);
        for (int c = 0; c < D / 64; ++c) ptx::tma_load_3d(S.k[st][c], &tm_k, &S.k_full[st], c * 64, kvh, k0);
        if (i >= NS && !ptx::mbar_wait(&S.v_empty[st], (use - 1) & 1, abort_flag, kWaitLimitNs)) {
          issued = -(i + 1);   // K of block i issued, V not
          break;
        }
        ptx::mbar_arrive_expect_tx(&S.v_full[st], D * 256);
        for (int c = 0; c < D / 64; ++c) ptx::tma_load_3d(S.v[st][c], &tm_v, &S.v_full[st], c * 64, kvh, k0);
        issued = i + 1;
      }
      if (*abort_flag) {
        // never leave a copy in flight into shared memory: wait (bounded, not
        // interruptible) for the last load of every stage and for Q
        const int last_k = issued < 0 ? -issued : issued;
        const int last_v = issued < 0 ? -issued - 1 : issued;
        for (int i = (last_k > NS ? last_k - NS : 0); i < last_k; ++i) ptx::mbar_drain(&S.k_full[i % NS], (i / NS) & 1);
        for (int i = (last_v > NS ? last_v - NS : 0); i < last_v; ++i) ptx::mbar_drain(&S.v_full[i % NS], (i / NS) & 1);
        ptx::mbar_drain(&S.q_full, 0);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (ptx::elect_one()) {
      constexpr uint32_t idesc_qk = ptx::idesc_bf16_f32(BM, kCols, false, false);
      constexpr uint32_t idesc_pv = ptx::idesc_bf16_f32(BM, D, false, true);
      bool ok = ptx::mbar_wait(kSplit ? &S.qt_full : &S.q_full, 0, abort_flag, kWaitLimitNs);
      ptx::tc_fence_after();
      // PV of one part (half the keys of S_s) of the keys kCols*hf.. of block
      // blk, so the first part's products run while the softmax still
      // computes the second part's P
      auto issue_pv = [&](int s, int blk, int hf, int part, bool first) {
        const uint32_t v_base = ptx::smem_addr(S.v[blk % NS][0]);
        const uint32_t o_col = tmem + cO0 + D * s;
        const uint32_t p_col = tmem + kCols * s;
        constexpr int kSteps = kCols / 32;   // 16-key steps per part
#pragma unroll
        for (int kk = part * kSteps; kk < (part + 1) * kSteps; ++kk) {
          // V block as the MN-major B operand: N = head dim (64-wide column
          // groups one box apart), K = 16 keys = 2 KB further per step
          const uint64_t bdesc =
              ptx::desc_add(ptx::sw128_desc(v_base, kBox, 1024), (kCols / 16 * hf + kk) * 2048);
          // P of this step: the part's columns start at part * kCols/2
          const uint32_t a = p_col + part * (kCols / 2) + (kk - part * kSteps) * 8;
          ptx::mma_ts(o_col, a, bdesc, idesc_pv, (!first || kk > 0) ? 1u : 0u);
          if constexpr (kHiLo) ptx::mma_ts(o_col, a + kCols / 4, bdesc, idesc_pv, 1u);
        }
      };
      // PV of slot s's n-th S (block blk, keys kCols*hf..), once both parts of its P are stored
      auto finish_pv = [&](int s, int blk, int hf, int n) {
        if (!ptx::mbar_wait(&S.p_half[s], n & 1, abort_flag, kWaitLimitNs)) return false;
        ptx::tc_fence_after();
        issue_pv(s, blk, hf, 0, n == 0);
        if (!ptx::mbar_wait(&S.p_full[s], n & 1, abort_flag, kWaitLimitNs)) return false;
        ptx::tc_fence_after();
        issue_pv(s, blk, hf, 1, n == 0);
        return true;
      };
      auto wait_v = [&](int blk) {
        return ptx::mbar_wait(&S.v_full[blk % NS], (blk / NS) & 1, abort_flag, kWaitLimitNs);
      };
      if constexpr (!kSplit) {
        // two heads: PV_0(i-1), S_0(i), PV_1(i-1), S_1(i); QK^T reads Q from
        // shared memory (TMEM holds the two S and two O accumulators)
        const uint32_t q_base[2] = {ptx::smem_addr(S.q[0][0]), ptx::smem_addr(S.q[HPC - 1][0])};
        for (int i = 0; ok && i < n_blocks; ++i) {
          const int st = i % NS;
          if (!ptx::mbar_wait(&S.k_full[st], (i / NS) & 1, abort_flag, kWaitLimitNs)) { ok = false; break; }
          ptx::tc_fence_after();
          const uint32_t k_base = ptx::smem_addr(S.k[st][0]);
          for (int s = 0; s < 2; ++s) {
            if (i > 0) {
              if (s == 0 && !wait_v(i - 1)) { ok = false; break; }
              if (!finish_pv(s, i - 1, 0, i - 1)) { ok = false; break; }
            }
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              // Q and K as K-major operands: 16 elements = 32 bytes per step
              // inside a 64-element box, next box after 4 steps
              const uint32_t koff = (kk >> 2) * kBox + (kk & 3) * 32;
              const uint64_t adesc = ptx::desc_add(ptx::sw128_desc(q_base[s], 16, 1024), koff);
              const uint64_t bdesc = ptx::desc_add(ptx::sw128_desc(k_base, 16, 1024), koff);
              ptx::mma_ss(tmem + kCols * s, adesc, bdesc, idesc_qk, kk > 0 ? 1u : 0u);
            }
            ptx::mma_commit(&S.s_full[s]);
          }
          if (!ok) break;
          ptx::mma_commit(&S.k_empty[st]);
          if (i > 0) ptx::mma_commit(&S.v_empty[(i - 1) % NS]);
        }
      } else {
        // one head: slot s takes keys 64s.. of every block; QK^T reads Q from
        // TMEM; a slot's PV is issued one block later, once its P is stored
        for (int i = 0; ok && i < n_blocks; ++i) {
          const int st = i % NS;
          if (!ptx::mbar_wait(&S.k_full[st], (i / NS) & 1, abort_flag, kWaitLimitNs)) { ok = false; break; }
          ptx::tc_fence_after();
          for (int s = 0; s < 2; ++s) {
            if (i > 0) {
              if (s == 0 && !wait_v(i - 1)) { ok = false; break; }
              if (!finish_pv(s, i - 1, s, i - 1)) { ok = false; break; }
            }
            const uint32_t k_base = ptx::smem_addr(S.k[st][0]) + s * (kBox / 2);   // key rows 64s..
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t koff = (kk >> 2) * kBox + (kk & 3) * 32;
              const uint64_t bdesc = ptx::desc_add(ptx::sw128_desc(k_base, 16, 1024), koff);
              ptx::mma_ts(tmem + kCols * s, tmem + cQ0 + kk * 8, bdesc, idesc_qk, kk > 0 ? 1u : 0u);
            }
            ptx::mma_commit(&S.s_full[s]);
          }
          if (!ok) break;
          ptx::mma_commit(&S.k_empty[st]);
          if (i > 0) ptx::mma_commit(&S.v_empty[(i - 1) % NS]);
        }
      }
      // the last block's PV products are still due
      if (ok && n_blocks > 0 && wait_v(n_blocks - 1)) {
        for (int s = 0; s < 2; ++s) {
          if (!finish_pv(s, n_blocks - 1, kSplit ? s : 0, n_blocks - 1)) break;
          ptx::mma_commit(&S.o_done[s]);
        }
      }
      // drain: every MMA issued above has completed before TMEM is released
      ptx::mma_commit(&S.drain);
      ptx::mbar_drain(&S.drain, 0);
    }
  }
  } else {
    // ------------------------------------------------------------ softmax
    ptx::regs_inc<kRegsSoftmax>();
    const int slot = (warp - 4) >> 2;
    const int wq = warp & 3;                 // TMEM lane quarter of this warp
    const int r = wq * 32 + (threadIdx.x & 31);
    const int qi = q0 + r;                   // this thread's query (forwarded index)
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t s_tm = tmem + lane_off + kCols * slot;
    const uint32_t o_tm = tmem + lane_off + cO0 + D * slot;
    const float sl2 = p.scale_log2;
    float m_used = -INFINITY;   // running maximum in use (log2 units)
    float l = 0.f;              // running row sum (relative to m_used)
    bool ok = true;
    if constexpr (kSplit) {
      // row r of the Q tile into TMEM lane r (the A operand of QK^T).  The
      // tile sits in shared memory as 128-byte-swizzled boxes of 64 elements
      // (16-byte chunk c of row r at chunk c ^ (r % 8)); TMEM column w holds
      // elements 2w, 2w+1.  The two warpgroups take alternate boxes.
      ok = ptx::mbar_wait(&S.q_full, 0, abort_flag, kWaitLimitNs);
      ok = __all_sync(0xffffffffu, ok);
      if (ok) {
#pragma unroll
        for (int b = 0; b < D / 64; ++b) {
          if ((b & 1) != slot) continue;
          uint32_t w[32];
          const uint8_t* row = S.q[0][b] + r * 128;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint4 v = *reinterpret_cast<const uint4*>(row + ((c ^ (r & 7)) << 4));
            w[4 * c] = v.x;
            w[4 * c + 1] = v.y;
            w[4 * c + 2] = v.z;
            w[4 * c + 3] = v.w;
          }
          ptx::tmem_st32(tmem + lane_off + cQ0 + b * 32, w);
        }
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        ptx::mbar_arrive(&S.qt_full);
      }
    }
    // two heads: every block, all its keys; one head: keys 64*slot.. of every block
    const int hf = kSplit ? slot : 0;
    int n_masked = 0;   // masked blocks so far (selects the subtree_end buffer)
    for (int jj = 0; ok && jj < n_blocks; ++jj) {
      ok = ptx::mbar_wait(&S.s_full[slot], jj & 1, abort_flag, kWaitLimitNs);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      ptx::tc_fence_after();
      const int2 blk = __ldg(&p.kb[kb_begin + jj]);
      const int k0 = blk.x + kCols * hf, nk = (blk.y & 0xFFFF) - kCols * hf;
      const bool full = (blk.y >> 16) & 1;
      float sv[kCols];
      {
        uint32_t u[kCols];
#pragma unroll
        for (int c = 0; c < kCols / 32; ++c)
          ptx::tmem_ld32(s_tm + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&u[c * 32]));
        ptx::tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < kCols; ++j) sv[j] = __uint_as_float(u[j]);
      }
      if (!full) {
        // key j = k0 + c is visible to query qi iff j <= qi < subtree_end[j].
        // The warpgroup stages the keys' subtree_end in shared memory (one
        // load per thread; 0 past the block's end, which hides the column),
        // meets at its se_bar (a bounded wait, like every wait here), then
        // every row tests all columns from there.  Two buffers by the parity
        // of the masked-block count: a buffer is rewritten only after every
        // thread of the warpgroup has arrived for the next masked block, i.e.
        // has finished reading it.
        int* se = S.se[slot][n_masked & 1];
        if (r < kCols) se[r] = r < nk ? __ldg(p.subtree_end + k0 + r) : 0;
        ptx::mbar_arrive(&S.se_bar[slot]);
        ok = ptx::mbar_wait(&S.se_bar[slot], n_masked & 1, abort_flag, kWaitLimitNs);
        ok = __all_sync(0xffffffffu, ok);
        ++n_masked;
        if (!ok) break;
        const int cmax = qi - k0;   // columns c <= cmax hold keys j <= qi
#pragma unroll
        for (int c = 0; c < kCols; c += 4) {
          const int4 e = ptx::lds128i(se + c);
          if (!(c <= cmax && qi < e.x)) sv[c] = -INFINITY;
          if (!(c + 1 <= cmax && qi < e.y)) sv[c + 1] = -INFINITY;
          if (!(c + 2 <= cmax && qi < e.z)) sv[c + 2] = -INFINITY;
          if (!(c + 3 <= cmax && qi < e.w)) sv[c + 3] = -INFINITY;
        }
      }
      // row maximum: 3-input max, four independent chains
      float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int c = 0; c < kCols; c += 8) {   // columns c .. c+7, exactly 0 .. kCols-1
#pragma unroll
        for (int x = 0; x < 4; ++x) m4[x] = ptx::max3(m4[x], sv[c + 2 * x], sv[c + 2 * x + 1]);
      }
      const float mx = ptx::max3(m4[0], m4[1], fmaxf(m4[2], m4[3]));
      const float m_blk = mx * sl2;
      float alpha = 1.f;
      const bool raise = m_blk > m_used + kRescaleThreshold;
      if (raise) {
        alpha = ptx::ex2(m_used - m_blk);   // 0 when m_used = -inf
        m_used = m_blk;
      }
      if (jj > 0 && __any_sync(0xffffffffu, raise)) {
        // O accumulated through this slot's previous block is complete: the
        // S commit this warp waited on tracks every earlier MMA, including
        // that block's PV.  It is rescaled before any P of this block is
        // released to the PV products.
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t u[32];
          ptx::tmem_ld32(o_tm + c * 32, u);
          ptx::tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 32; ++j) u[j] = __float_as_uint(__uint_as_float(u[j]) * alpha);
          ptx::tmem_st32(o_tm + c * 32, u);
        }
      }
      const float m_sub = (m_used == -INFINITY) ? 0.f : m_used;
      // exponent arguments and the row sum on packed fp32 pairs; P of the
      // first half of the keys is released (p_half) before the second half
      // is computed
      const uint64_t sl2x2 = ptx::f2(sl2, sl2), negm = ptx::f2(-m_sub, -m_sub);
      uint64_t sum2[2] = {0ull, 0ull};
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t pk[kCols / 4];
        uint32_t pl[kHiLo ? kCols / 4 : 1];
#pragma unroll
        for (int j = 0; j < kCols / 4; ++j) {
          float a0, a1;
          ptx::unf2(ptx::fma2(ptx::f2(sv[c * (kCols / 2) + 2 * j], sv[c * (kCols / 2) + 2 * j + 1]), sl2x2, negm),
                    a0, a1);
          const float p0 = ptx::ex2(a0), p1 = ptx::ex2(a1);
          sum2[j & 1] = ptx::add2(sum2[j & 1], ptx::f2(p0, p1));
          if constexpr (kHiLo)
            ptx::split_bf16x2(p0, p1, pk[j], pl[j]);
          else
            pk[j] = ptx::pack_bf16x2(p0, p1);
        }
        // part c at column c * kCols/2 (every S column was read above); the
        // precise mode's low halves kCols/4 further
        if constexpr (kCols == 128) {
          ptx::tmem_st32(s_tm + c * 64, pk);
          if constexpr (kHiLo) ptx::tmem_st32(s_tm + c * 64 + 32, pl);
        } else {
          ptx::tmem_st16(s_tm + c * 32, pk);
          if constexpr (kHiLo) ptx::tmem_st16(s_tm + c * 32 + 16, pl);
        }
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        ptx::mbar_arrive(c == 0 ? &S.p_half[slot] : &S.p_full[slot]);
      }
      float s0, s1, s2, s3;
      ptx::unf2(sum2[0], s0, s1);
      ptx::unf2(sum2[1], s2, s3);
      const float sum = (s0 + s1) + (s2 + s3);
      l = l * alpha + sum;
    }
    if constexpr (kSplit) {
      // one head: merge the two slots' partial results row by row
      if (ok) {
        S.mrg[slot][0][r] = m_used;
        S.mrg[slot][1][r] = l;
        ptx::mbar_arrive(&S.mrg_bar);
        ok = ptx::mbar_wait(&S.mrg_bar, 0, abort_flag, kWaitLimitNs) &&
             ptx::mbar_wait(&S.o_done[0], 0, abort_flag, kWaitLimitNs) &&
             ptx::mbar_wait(&S.o_done[1], 0, abort_flag, kWaitLimitNs);
        ok = __all_sync(0xffffffffu, ok);
      }
      if (ok) {
        ptx::tc_fence_after();
        const float m0 = S.mrg[0][0][r], l0 = S.mrg[0][1][r], m1 = S.mrg[1][0][r], l1 = S.mrg[1][1][r];
        const float m = fmaxf(m0, m1);
        const float c0 = m0 == -INFINITY ? 0.f : ptx::ex2(m0 - m);
        const float c1 = m1 == -INFINITY ? 0.f : ptx::ex2(m1 - m);
        const float lt = l0 * c0 + l1 * c1;
        const float inv = lt > 0.f ? 1.f / lt : 0.f;
        const float w0 = c0 * inv, w1 = c1 * inv;
        // this warpgroup writes half of the head dimension from both O
        const uint32_t oa = tmem + lane_off + cO0 + (D / 2) * slot, ob = oa + D;
        __nv_bfloat16* orow = p.o + (static_cast<int64_t>(qi) * p.Hq + h0) * D + (D / 2) * slot;
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
          uint32_t ua[32], ub[32];
          ptx::tmem_ld32(oa + c * 32, ua);
          ptx::tmem_ld32(ob + c * 32, ub);
          ptx::tmem_wait_ld();
          if (r < nq) {
            uint32_t pk[16], pl[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const float x0 = __uint_as_float(ua[2 * j]) * w0 + __uint_as_float(ub[2 * j]) * w1;
              const float x1 = __uint_as_float(ua[2 * j + 1]) * w0 + __uint_as_float(ub[2 * j + 1]) * w1;
              if constexpr (kHiLo)
                ptx::split_bf16x2(x0, x1, pk[j], pl[j]);
              else
                pk[j] = ptx::pack_bf16x2(x0, x1);
            }
            uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
            for (int j = 0; j < 4; ++j) dst[j] = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
            if (kHiLo && p.o_lo) {
              uint4* dlo = reinterpret_cast<uint4*>(p.o_lo + (orow - p.o) + c * 32);
#pragma unroll
              for (int j = 0; j < 4; ++j) dlo[j] = make_uint4(pl[4 * j], pl[4 * j + 1], pl[4 * j + 2], pl[4 * j + 3]);
            }
          }
        }
        if (r < nq && slot == 0) {
          const float lse = lt > 0.f ? (m + log2f(lt)) * 0.69314718055994530942f : -INFINITY;
          p.lse[static_cast<int64_t>(h0) * p.F + qi] = lse;
        }
      }
    } else {
    if (ok) {
      ok = ptx::mbar_wait(&S.o_done[slot], 0, abort_flag, kWaitLimitNs);
      ok = __all_sync(0xffffffffu, ok);
    }
    if (ok) {
      ptx::tc_fence_after();
      const int h = h0 + slot;
      const float inv_l = l > 0.f ? 1.f / l : 0.f;
      __nv_bfloat16* orow = p.o + (static_cast<int64_t>(qi) * p.Hq + h) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t u[32];
        ptx::tmem_ld32(o_tm + c * 32, u);
        ptx::tmem_wait_ld();
        if (r < nq) {
          uint32_t pk[16], pl[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float x0 = __uint_as_float(u[2 * j]) * inv_l, x1 = __uint_as_float(u[2 * j + 1]) * inv_l;
            if constexpr (kHiLo)
              ptx::split_bf16x2(x0, x1, pk[j], pl[j]);
            else
              pk[j] = ptx::pack_bf16x2(x0, x1);
          }
          uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
          for (int j = 0; j < 4; ++j) dst[j] = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
          if (kHiLo && p.o_lo) {
            uint4* dlo = reinterpret_cast<uint4*>(p.o_lo + (orow - p.o) + c * 32);
#pragma unroll
            for (int j = 0; j < 4; ++j) dlo[j] = make_uint4(pl[4 * j], pl[4 * j + 1], pl[4 * j + 2], pl[4 * j + 3]);
          }
        }
      }
      if (r < nq) {
        const float lse = l > 0.f ? (m_used + log2f(l)) * 0.69314718055994530942f : -INFINITY;
        p.lse[static_cast<int64_t>(h) * p.F + qi] = lse;
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

template <int D, int HPC, int NS, bool kHiLo>
int launch(const FwdParams& prm, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, int64_t items,
           cudaStream_t stream) {
  auto kern = tree_attn_fwd_kernel<D, HPC, NS, kHiLo>;
  constexpr size_t smem = fwd_smem_bytes<D, HPC, NS>();
  static_assert(smem <= 227 * 1024, "shared memory");
  // the shared-memory limit is an attribute of the kernel in one context, so
  // it is set once per context (per device), not once per process
  static PerContext<int> configured;
  int unused = 0;
  const int st = configured.get(&unused, [&](int*) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
        cudaSuccess)
      return TPK_E_CUDA;
    // the warpgroups' register shares must fit in what the CTA launches with
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess) return TPK_E_CUDA;
    if (fa.numRegs * 384 < kRegsNeeded) return TPK_E_UNSUPPORTED;
    return TPK_OK;
  });
  if (st != TPK_OK) return st;
  if (items <= 0) return TPK_OK;
  if (items > 0x7fffffff) return TPK_E_OVERFLOW;
  kern<<<static_cast<unsigned>(items), 384, smem, stream>>>(tq, tk, tv, prm);
  return cuda_status(cudaGetLastError());
}

template <bool kHiLo>
int launch_all(int d, int hpc, const FwdParams& prm, const CUtensorMap& tq, const CUtensorMap& tk,
               const CUtensorMap& tv, int64_t items, cudaStream_t s) {
  if (d == 128)
    return hpc == 2 ? launch<128, 2, 2, kHiLo>(prm, tq, tk, tv, items, s) : launch<128, 1, 2, kHiLo>(prm, tq, tk, tv, items, s);
  return hpc == 2 ? launch<64, 2, 3, kHiLo>(prm, tq, tk, tv, items, s) : launch<64, 1, 4, kHiLo>(prm, tq, tk, tv, items, s);
}

}  // namespace
}  // namespace tpk

extern "C" int tpk_tree_attn_fwd_ex(const tpk_plan* plan, const void* dev_image, const void* q, const void* k,
                                    const void* v, void* o, float* lse, int32_t Hq, int32_t Hkv, int32_t d,
                                    float scale, const tpk_attn_opts* opts, int32_t* dev_err, void* stream) {
  using namespace tpk;
  if (!plan || !dev_image || !q || !k || !v || !o || !lse) return TPK_E_ARG;
  if (Hq <= 0 || Hkv <= 0 || !(scale > 0.f)) return TPK_E_ARG;
  if ((d != 64 && d != 128) || Hq % Hkv != 0) return TPK_E_UNSUPPORTED;
  if (opts && ((opts->precision != TPK_PREC_FAST && opts->precision != TPK_PREC_PRECISE) || opts->rope_base != 0.0))
    return TPK_E_ARG;
  const bool precise = opts && opts->precision == TPK_PREC_PRECISE;
  void* o_lo = precise ? opts->o_lo : nullptr;
  if ((reinterpret_cast<uintptr_t>(o) | reinterpret_cast<uintptr_t>(o_lo) | reinterpret_cast<uintptr_t>(dev_image) % 256) %
      16)
    return TPK_E_ARG;
  const Plan& P = plan->p;
  if (P.F == 0) return TPK_OK;
  int st = check_device();
  if (st != TPK_OK) return st;
  CUtensorMap tq, tk, tv;
  if ((st = make_map_bf16(&tq, q, P.F, Hq, d, 128)) != TPK_OK) return st;
  if ((st = make_map_bf16(&tk, k, P.F, Hkv, d, 128)) != TPK_OK) return st;
  if ((st = make_map_bf16(&tv, v, P.F, Hkv, d, 128)) != TPK_OK) return st;
  const uint8_t* img = static_cast<const uint8_t*>(dev_image);
  FwdParams prm;
  prm.qt_q0 = reinterpret_cast<const int32_t*>(img + P.off_qt_q0);
  prm.qt_nq = reinterpret_cast<const int32_t*>(img + P.off_qt_nq);
  prm.qt_kb_begin = reinterpret_cast<const int32_t*>(img + P.off_qt_kb_begin);
  prm.kb = reinterpret_cast<const int2*>(img + P.off_kb);
  prm.qt_order = reinterpret_cast<const int32_t*>(img + P.off_qt_order);
  prm.subtree_end = reinterpret_cast<const int32_t*>(img + P.off_subtree_end);
  prm.o = static_cast<__nv_bfloat16*>(o);
  prm.o_lo = static_cast<__nv_bfloat16*>(o_lo);
  prm.lse = lse;
  prm.F = static_cast<int32_t>(P.F);
  prm.Hq = Hq;
  prm.group_size = Hq / Hkv;
  prm.scale_log2 = scale * 1.4426950408889634f;
  prm.err = dev_err;
  const int hpc = (prm.group_size % 2 == 0) ? 2 : 1;
  prm.n_hgroups = Hq / hpc;
  const int64_t items = static_cast<int64_t>(P.qt_q0.size()) * prm.n_hgroups;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return precise ? launch_all<true>(d, hpc, prm, tq, tk, tv, items, s) : launch_all<false>(d, hpc, prm, tq, tk, tv, items, s);
}

extern "C" int tpk_tree_attn_fwd(const tpk_plan* plan, const void* dev_image, const void* q, const void* k,
                                 const void* v, void* o, float* lse, int32_t Hq, int32_t Hkv, int32_t d, float scale,
                                 void* workspace, size_t ws_bytes, int32_t* dev_err, void* stream) {
  (void)workspace;
  (void)ws_bytes;
  return tpk_tree_attn_fwd_ex(plan, dev_image, q, k, v, o, lse, Hq, Hkv, d, scale, nullptr, dev_err, stream);
}
