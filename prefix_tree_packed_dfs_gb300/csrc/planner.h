// Host-side packing planner: prefix tree, row placement, depth-first layout and
// the attention kernels' work lists.  Integer-only ("Prefix Tree Packing in
// ART", section "Metadata space first": the plan is computed over plain
// integers before any tensor is touched).
#pragma once
#include <cstdint>
#include <cstddef>
#include <memory>
#include <new>
#include <utility>
#include <vector>

namespace tpk {

// Allocator whose resize() leaves new elements uninitialised: for a buffer
// that is written in full right after it is sized (the device image).
template <typename T>
struct UninitAllocator : std::allocator<T> {
  template <typename U>
  struct rebind {
    using other = UninitAllocator<U>;
  };
  UninitAllocator() noexcept = default;
  template <typename U>
  UninitAllocator(const UninitAllocator<U>&) noexcept {}
  template <typename U>
  void construct(U* p) noexcept {
    ::new (static_cast<void*>(p)) U;
  }
  template <typename U, typename... A>
  void construct(U* p, A&&... a) {
    ::new (static_cast<void*>(p)) U(std::forward<A>(a)...);
  }
};

constexpr int kTile = 128;   // query / key tile height of the attention kernels

struct PlanOptions {
  int64_t row_capacity = 65536;
  int32_t min_shared = 64;
  int32_t placement = 0;     // 0 best-fit decreasing, 1 next-fit
};

struct Plan {
  // sizes
  int64_t n_seqs = 0, R = 0, F = 0, n_rows = 0, n_segments = 0, n_leaves = 0;
  int64_t useful_pairs = 0, visited_pairs = 0, max_depth = 0;
  double packing_ratio = 0, row_fill_frac = 0, fork_frac = 0;
  int64_t row_capacity = 0;

  // layout
  std::vector<int64_t> row_offsets, row_loads;
  std::vector<int32_t> row_of_seq, fwd_token, fwd_src, parent, depth, token_index, subtree_end;
  // raw tokens of each forwarded position (the inverse of token_index, CSR):
  // fwd_raw[fwd_raw_begin[f] .. fwd_raw_begin[f+1]) ascending, first = fwd_src[f]
  std::vector<int32_t> fwd_raw_begin, fwd_raw;

  // forward work list: query tiles and their key blocks
  std::vector<int32_t> qt_q0, qt_nq, qt_kb_begin, kb, qt_order;
  // backward work list: key tiles and their query blocks
  std::vector<int32_t> kt_k0, kt_nk, kt_qb_begin, qb, kt_order;
  // segment instances (a segment placed in one row) by tree level:
  // instances [seg_level_begin[l], seg_level_begin[l+1]) are level l; each
  // covers forwarded [seg_start, +seg_len); seg_parent indexes this order;
  // seg_off = positions of the instances before it on its level (scratch
  // offsets of a level-by-level pass)
  std::vector<int32_t> seg_level_begin, seg_start, seg_len, seg_parent, seg_off;

  // device image: every array above that a kernel reads, 256-byte aligned sections
  std::vector<uint8_t, UninitAllocator<uint8_t>> image;
  size_t off_depth = 0, off_token_index = 0, off_subtree_end = 0, off_parent = 0;
  size_t off_fwd_raw_begin = 0, off_fwd_raw = 0;
  size_t off_qt_q0 = 0, off_qt_nq = 0, off_qt_kb_begin = 0, off_kb = 0, off_qt_order = 0;
  size_t off_kt_k0 = 0, off_kt_nk = 0, off_kt_qb_begin = 0, off_qb = 0, off_kt_order = 0;
  size_t off_seg_start = 0, off_seg_len = 0, off_seg_parent = 0, off_seg_off = 0;

  // Back to an empty plan, keeping every array's allocation: a plan built
  // into recycled storage writes into memory that is already mapped.  Every
  // member above is reset here.
  void reset_keep_capacity() {
    n_seqs = R = F = n_rows = n_segments = n_leaves = 0;
    useful_pairs = visited_pairs = max_depth = 0;
    packing_ratio = row_fill_frac = fork_frac = 0;
    row_capacity = 0;
    row_offsets.clear();
    row_loads.clear();
    for (std::vector<int32_t>* v : {&row_of_seq, &fwd_token, &fwd_src, &parent, &depth, &token_index, &subtree_end,
                                    &fwd_raw_begin, &fwd_raw, &qt_q0, &qt_nq, &qt_kb_begin, &kb, &qt_order, &kt_k0,
                                    &kt_nk, &kt_qb_begin, &qb, &kt_order, &seg_level_begin, &seg_start, &seg_len,
                                    &seg_parent, &seg_off})
      v->clear();
    image.clear();
    off_depth = off_token_index = off_subtree_end = off_parent = 0;
    off_fwd_raw_begin = off_fwd_raw = 0;
    off_qt_q0 = off_qt_nq = off_qt_kb_begin = off_kb = off_qt_order = 0;
    off_kt_k0 = off_kt_nk = off_kt_qb_begin = off_qb = off_kt_order = 0;
    off_seg_start = off_seg_len = off_seg_parent = off_seg_off = 0;
  }
};

// Returns a TPK_* status; on success fills *out.
int build_plan(const int32_t* tokens, const int64_t* seq_offsets, int32_t n_seqs,
               const uint8_t* trained, const int32_t* group_ids,
               const PlanOptions& opts, Plan* out);

}  // namespace tpk
