// Host packing planner.  Integer-only; no CUDA.
//
// Steps ("Prefix Tree Packing in ART" = [ART], "DAG packing" = [DAG],
// "TRL Tree Packing for AsyncGRPO" = [TRL]):
//  1. position symbols (token, trained flag, target-if-trained): two positions
//     share one forwarded slot iff their symbol prefixes agree, which keeps the
//     last common token once per branch ([ART] "The tree", off-by-one note;
//     [DAG] "The walk": the last common node is copied for every child);
//  2. the prefix tree.  [ART] "The tree" builds it by a recursive walk
//     (longest run all active sequences agree on, emit once, split by the next
//     symbol).  Here the same tree comes from sorting the sequences'
//     symbol strings and taking adjacent longest-common-prefix lengths: the
//     sequences under any tree node are a contiguous run of the sorted order,
//     the node's shared run ends at the minimum adjacent LCP inside that run,
//     and the children are the sub-runs separated where the LCP equals it.
//     Shared runs shorter than min_shared are not emitted; their positions
//     are carried into each child ([ART] "The tree", first refinement);
//  3. placement of leaves into rows: best-fit decreasing over marginal cost
//     ([ART] "Bin packing, with a twist"), next-fit ([ART] "One tree, not one
//     per group") or one row per placement group (no counterpart on the pages:
//     a data-parallel rank rebuilding the rows it owns); a row's segment set
//     is closed under ancestors, so a leaf's marginal cost is the length of
//     its path below the deepest segment the row already holds;
//  4. depth-first layout of each row (leaves in symbol order, each segment
//     emitted once, parents first; [DAG] "The walk", [TRL] "How tree packing
//     works"), depth positions ([DAG] "Positions"), token_index, subtree ends
//     ([ART] "Token-mixing layers": [enter, exit] intervals);
//  5. the kernels' work lists: per 128-query tile, the key blocks of the
//     ancestor chain of its first query plus the tile itself; per 128-key tile,
//     the query blocks of [k0, max subtree_end).  Launch order: runs of
//     kOrderChunk consecutive tiles (depth-first order, so neighbouring
//     subtrees), runs in decreasing total work, tiles of a run longest first.
//     CTAs resident at the same time then read the same ancestor K/V blocks
//     (query tiles) or descendant Q/dO blocks (key tiles) and share them in
//     L2, while long work still starts before short work.
// Host threads: symbols per sequence, the symbol-string sort in chunks
// (merged stably), and layout, subtree ends, work lists and raw-token lists
// per row -- once rows are placed, each row's forwarded range and instance
// range are fixed, tiles read only their row and a row holds only its own
// sequences' raw tokens -- each write only their own outputs, so the plan
// does not depend on the thread count.  The caller may hand in the storage
// of an earlier plan (Plan::reset_keep_capacity) to skip fresh allocations.
#include "planner.h"

#include <algorithm>
#include <atomic>
#include <cstdlib>
#include <cstring>
#include <exception>
#include <limits>
#include <mutex>
#include <numeric>
#include <system_error>
#include <thread>
#include <unordered_map>

#include "tpk.h"

namespace tpk {
namespace {

constexpr int64_t kNoTarget = -2;  // untrained position: target not part of the key
constexpr int64_t kEos = -1;       // target of the last position
constexpr int32_t kOrderChunk = 128;   // tiles per run of the launch order (16384 tokens)

inline uint64_t pack_symbol(int32_t token, int flag, int64_t target) {
  // lexicographic (token, flag, target) as one unsigned integer: tokens are
  // >= 0 (31 bits), flag 1 bit, target + 2 in [0, 2^31 + 1] (32 bits)
  return (static_cast<uint64_t>(static_cast<uint32_t>(token)) << 33) |
         (static_cast<uint64_t>(flag ? 1 : 0) << 32) |
         static_cast<uint64_t>(target + 2);
}

struct Segment {
  int32_t parent;
  int32_t start;   // depth of the first position
  int32_t end;     // one past the depth of the last position
  int32_t n_children;
};

struct Leaf {
  std::vector<int32_t> members;   // original sequence indices, ascending
  std::vector<int32_t> path;      // segment ids, root first
  int32_t rank;                   // position of the sequence in symbol order
  int64_t cost;                   // standalone cost = sequence length
  int32_t rep() const { return members.front(); }
};

struct Bin {
  int64_t load = 0;
  std::vector<int32_t> leaves;
  std::vector<uint64_t> held;     // bitset over segments
  bool has(int32_t s) const { return (held[s >> 6] >> (s & 63)) & 1; }
  void set(int32_t s) { held[s >> 6] |= (uint64_t{1} << (s & 63)); }
};

int64_t marginal_cost(const Bin& b, const Leaf& leaf, const std::vector<Segment>& segs) {
  int64_t c = 0;
  for (size_t i = leaf.path.size(); i-- > 0;) {
    int32_t s = leaf.path[i];
    if (b.has(s)) break;   // everything above is held too
    c += segs[s].end - segs[s].start;
  }
  return c;
}

void take(Bin& b, int32_t leaf_id, const Leaf& leaf, const std::vector<Segment>& segs) {
  b.load += marginal_cost(b, leaf, segs);
  for (int32_t s : leaf.path) b.set(s);
  b.leaves.push_back(leaf_id);
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Host threads the planner may use: TPK_PLANNER_THREADS if set (>= 1), else
// the hardware's, at most 16.
int64_t planner_threads() {
  const char* env = std::getenv("TPK_PLANNER_THREADS");
  if (env && std::atoll(env) >= 1) return std::min<int64_t>(std::atoll(env), 16);
  return std::min<int64_t>(std::max<int64_t>(1, std::thread::hardware_concurrency()), 16);
}

// fn(i) for i in [0, n) on the planner's host threads; every i writes only
// its own outputs, so the result does not depend on the schedule.
// An exception thrown by fn on any thread (std::bad_alloc, say) stops the
// remaining indices from being started and is rethrown on the calling thread
// after every worker has joined, so it reaches the C ABI's handler instead of
// terminating the process.  If a worker thread cannot be created (a process
// or container thread limit), the threads that exist -- at least the calling
// one -- take the remaining indices.
template <typename Fn>
void parallel_for(int64_t n, Fn fn) {
  const int64_t nt = std::min<int64_t>(planner_threads(), n);
  if (nt <= 1) {
    for (int64_t i = 0; i < n; ++i) fn(i);
    return;
  }
  std::atomic<int64_t> next{0};
  std::mutex err_mu;
  std::exception_ptr err;
  auto worker = [&]() {
    try {
      for (int64_t i; (i = next.fetch_add(1, std::memory_order_relaxed)) < n;) fn(i);
    } catch (...) {
      next.store(n, std::memory_order_relaxed);   // no new indices after a failure
      std::lock_guard<std::mutex> lock(err_mu);
      if (!err) err = std::current_exception();
    }
  };
  std::vector<std::thread> pool;
  try {
    pool.reserve(static_cast<size_t>(nt - 1));
    for (int64_t t = 1; t < nt; ++t) pool.emplace_back(worker);
  } catch (const std::system_error&) {
    // fewer threads than asked for: the ones started and this one share the work
  } catch (const std::bad_alloc&) {
  }
  worker();
  for (auto& th : pool) th.join();
  if (err) std::rethrow_exception(err);
}

// std::stable_sort of v by comp, on up to 16 host threads: contiguous chunks
// are sorted stably in parallel, then neighbours are merged stably in rounds
// (the left range's elements first among equals), which gives exactly the
// permutation a single stable sort gives.
template <typename Comp>
void parallel_stable_sort(std::vector<int32_t>& v, Comp comp) {
  const int64_t n = static_cast<int64_t>(v.size());
  const int64_t chunks = std::min<int64_t>(planner_threads(), n / 64);
  if (chunks <= 1) {
    std::stable_sort(v.begin(), v.end(), comp);
    return;
  }
  std::vector<int64_t> cut(static_cast<size_t>(chunks) + 1);
  for (int64_t c = 0; c <= chunks; ++c) cut[c] = n * c / chunks;
  parallel_for(chunks, [&](int64_t c) { std::stable_sort(v.begin() + cut[c], v.begin() + cut[c + 1], comp); });
  while (cut.size() > 2) {
    const int64_t pairs = static_cast<int64_t>(cut.size() - 1) / 2;
    parallel_for(pairs, [&](int64_t i) {
      std::inplace_merge(v.begin() + cut[2 * i], v.begin() + cut[2 * i + 1], v.begin() + cut[2 * i + 2], comp);
    });
    std::vector<int64_t> next;
    for (size_t i = 0; i < cut.size(); i += 2) next.push_back(cut[i]);
    if (next.back() != cut.back()) next.push_back(cut.back());
    cut.swap(next);
  }
}

}  // namespace

int build_plan(const int32_t* tokens, const int64_t* seq_offsets, int32_t n_seqs,
               const uint8_t* trained, const int32_t* group_ids,
               const PlanOptions& opts, Plan* out) {
  if (!tokens || !seq_offsets || !out || n_seqs <= 0) return TPK_E_ARG;
  if (opts.row_capacity <= 0) return TPK_E_ARG;
  if (opts.placement != TPK_PLACE_BFD && opts.placement != TPK_PLACE_NEXT_FIT && opts.placement != TPK_PLACE_GROUPS)
    return TPK_E_ARG;
  if (seq_offsets[0] != 0) return TPK_E_ARG;
  for (int32_t s = 0; s < n_seqs; ++s)
    if (seq_offsets[s + 1] <= seq_offsets[s]) return TPK_E_ARG;
  const int64_t R = seq_offsets[n_seqs];
  if (R >= (int64_t{1} << 31)) return TPK_E_OVERFLOW;
  for (int64_t r = 0; r < R; ++r)
    if (tokens[r] < 0) return TPK_E_ARG;
  for (int32_t s = 0; s < n_seqs; ++s)
    if (seq_offsets[s + 1] - seq_offsets[s] > opts.row_capacity) return TPK_E_SEQ_TOO_LONG;

  Plan& P = *out;
  P.reset_keep_capacity();
  P.n_seqs = n_seqs;
  P.R = R;
  P.row_capacity = opts.row_capacity;
  auto len = [&](int32_t s) { return static_cast<int32_t>(seq_offsets[s + 1] - seq_offsets[s]); };

  // ---- 1. symbols --------------------------------------------------------
  std::vector<uint64_t, UninitAllocator<uint64_t>> sym(R);   // every element written below
  parallel_for(n_seqs, [&](int64_t si) {
    const int32_t s = static_cast<int32_t>(si);
    const int64_t o = seq_offsets[s];
    const int32_t L = len(s);
    for (int32_t p = 0; p < L; ++p) {
      const int flag = trained ? (trained[o + p] != 0) : 1;
      int64_t target = kNoTarget;
      if (flag || p == L - 1) target = (p + 1 < L) ? tokens[o + p + 1] : kEos;
      sym[o + p] = pack_symbol(tokens[o + p], flag, target);
    }
  });

  // ---- 2. tree -----------------------------------------------------------
  std::vector<int32_t> order(n_seqs);
  std::iota(order.begin(), order.end(), 0);
  parallel_stable_sort(order, [&](int32_t a, int32_t b) {
    return std::lexicographical_compare(sym.begin() + seq_offsets[a], sym.begin() + seq_offsets[a + 1],
                                        sym.begin() + seq_offsets[b], sym.begin() + seq_offsets[b + 1]);
  });
  std::vector<int32_t> rank(n_seqs);
  for (int32_t i = 0; i < n_seqs; ++i) rank[order[i]] = i;
  std::vector<int32_t> lcp(n_seqs, 0);   // lcp[i]: common prefix of order[i-1], order[i]
  for (int32_t i = 1; i < n_seqs; ++i) {
    const int32_t a = order[i - 1], b = order[i];
    const int32_t n = std::min(len(a), len(b));
    auto pa = sym.begin() + seq_offsets[a];
    auto pb = sym.begin() + seq_offsets[b];
    lcp[i] = static_cast<int32_t>(std::mismatch(pa, pa + n, pb).first - pa);
  }

  std::vector<Segment> segs;
  std::vector<Leaf> leaves;
  const int32_t min_len = std::max<int32_t>(opts.min_shared, 1);
  struct Frame { int32_t lo, hi, seg_start, parent; };
  std::vector<Frame> stack{{0, n_seqs, 0, -1}};
  auto emit = [&](int32_t parent, int32_t start, int32_t end) {
    segs.push_back({parent, start, end, 0});
    if (parent >= 0) segs[parent].n_children++;
    return static_cast<int32_t>(segs.size() - 1);
  };
  while (!stack.empty()) {
    Frame fr = stack.back();
    stack.pop_back();
    bool identical = true;
    int32_t end = std::numeric_limits<int32_t>::max();
    for (int32_t i = fr.lo + 1; i < fr.hi; ++i) {
      end = std::min(end, lcp[i]);
      if (!(lcp[i] == len(order[i]) && len(order[i]) == len(order[i - 1]))) identical = false;
    }
    if (identical) {   // one distinct sequence: a leaf
      const int32_t L = len(order[fr.lo]);
      Leaf leaf;
      const int32_t sid = emit(fr.parent, fr.seg_start, L);
      for (int32_t i = fr.lo; i < fr.hi; ++i) leaf.members.push_back(order[i]);
      std::sort(leaf.members.begin(), leaf.members.end());
      for (int32_t s = sid; s >= 0; s = segs[s].parent) leaf.path.push_back(s);
      std::reverse(leaf.path.begin(), leaf.path.end());
      leaf.rank = fr.lo;
      leaf.cost = L;
      leaves.push_back(std::move(leaf));
      continue;
    }
    int32_t parent = fr.parent, seg_start = fr.seg_start;
    if (end > seg_start && end - seg_start >= min_len) {
      parent = emit(parent, seg_start, end);
      seg_start = end;
    }
    // children: sub-runs split where the adjacent LCP equals `end`; pushed in
    // reverse so the smallest symbol is walked first (depth first)
    int32_t hi = fr.hi;
    for (int32_t i = fr.hi - 1; i >= fr.lo; --i) {
      if (i == fr.lo || lcp[i] == end) {
        stack.push_back({i, hi, seg_start, parent});
        hi = i;
      }
    }
  }
  P.n_segments = static_cast<int64_t>(segs.size());
  P.n_leaves = static_cast<int64_t>(leaves.size());

  // ---- 3. placement -------------------------------------------------------
  std::vector<int32_t> by_input(leaves.size());
  std::iota(by_input.begin(), by_input.end(), 0);
  std::sort(by_input.begin(), by_input.end(),
            [&](int32_t a, int32_t b) { return leaves[a].rep() < leaves[b].rep(); });
  std::vector<std::vector<int32_t>> groups;   // in first-appearance order
  std::vector<int64_t> group_key;             // the id of each group
  {
    std::unordered_map<int64_t, size_t> index;
    for (int32_t li : by_input) {
      const int64_t g = group_ids ? group_ids[leaves[li].rep()] : leaves[li].path.front();
      auto it = index.find(g);
      if (it == index.end()) {
        it = index.emplace(g, groups.size()).first;
        groups.emplace_back();
        group_key.push_back(g);
      }
      groups[it->second].push_back(li);
    }
  }
  const int64_t C = opts.row_capacity;
  const size_t words = (segs.size() + 63) / 64;
  std::vector<Bin> bins;
  auto new_bin = [&]() { bins.emplace_back(); bins.back().held.assign(words, 0); return bins.size() - 1; };
  if (opts.placement == TPK_PLACE_BFD) {
    std::vector<int64_t> gmax(groups.size(), 0);
    for (size_t g = 0; g < groups.size(); ++g)
      for (int32_t li : groups[g]) gmax[g] = std::max(gmax[g], leaves[li].cost);
    std::vector<int32_t> gorder(groups.size());
    std::iota(gorder.begin(), gorder.end(), 0);
    std::stable_sort(gorder.begin(), gorder.end(), [&](int32_t a, int32_t b) { return gmax[a] > gmax[b]; });
    for (int32_t g : gorder) {
      for (int32_t li : groups[g]) {
        int64_t best = -1, best_room = C + 1;
        for (size_t b = 0; b < bins.size(); ++b) {
          const int64_t load = bins[b].load + marginal_cost(bins[b], leaves[li], segs);
          if (load <= C && C - load < best_room) { best = static_cast<int64_t>(b); best_room = C - load; }
        }
        if (best < 0) best = static_cast<int64_t>(new_bin());
        take(bins[best], li, leaves[li], segs);
      }
    }
  } else if (opts.placement == TPK_PLACE_GROUPS) {
    // one row per group, rows in increasing group id
    std::vector<int32_t> gorder(groups.size());
    std::iota(gorder.begin(), gorder.end(), 0);
    std::sort(gorder.begin(), gorder.end(), [&](int32_t a, int32_t b) { return group_key[a] < group_key[b]; });
    for (int32_t g : gorder) {
      const size_t b = new_bin();
      for (int32_t li : groups[g]) take(bins[b], li, leaves[li], segs);
      if (bins[b].load > C) return TPK_E_SEQ_TOO_LONG;
    }
  } else {
    for (auto& g : groups)
      for (int32_t li : g) {
        if (bins.empty() || bins.back().load + marginal_cost(bins.back(), leaves[li], segs) > C) new_bin();
        take(bins.back(), li, leaves[li], segs);
      }
  }
  P.n_rows = static_cast<int64_t>(bins.size());

  // ---- 4. layout ----------------------------------------------------------
  // Rows are laid out independently: row b fills the forwarded positions
  // [fbase[b], fbase[b+1]) (its load) and the segment instances (a segment
  // placed in one row) [ibase[b], ibase[b+1]) (its distinct segments), in
  // the same order as one sequential pass over the rows would.
  const size_t nb = bins.size();
  std::vector<int64_t> fbase(nb + 1, 0), ibase(nb + 1, 0);
  for (size_t b = 0; b < nb; ++b) {
    int64_t distinct = 0;
    for (const uint64_t w : bins[b].held) distinct += __builtin_popcountll(w);
    fbase[b + 1] = fbase[b] + bins[b].load;
    ibase[b + 1] = ibase[b] + distinct;
  }
  const int64_t F = fbase[nb];
  if (F >= (int64_t{1} << 31)) return TPK_E_OVERFLOW;
  P.F = F;
  P.depth.resize(F);
  P.fwd_token.resize(F);
  P.parent.resize(F);
  P.token_index.assign(R, -1);
  P.row_of_seq.assign(n_seqs, -1);
  P.row_offsets.assign(fbase.begin(), fbase.end());
  P.row_loads.resize(nb);
  for (size_t b = 0; b < nb; ++b) P.row_loads[b] = bins[b].load;
  std::vector<int32_t> inst_start(ibase[nb]), inst_len(ibase[nb]), inst_parent(ibase[nb]);
  std::vector<int32_t, UninitAllocator<int32_t>> inst_of(F);   // every position written by its row
  parallel_for(static_cast<int64_t>(nb), [&](int64_t bi) {
    const size_t b = static_cast<size_t>(bi);
    std::vector<int32_t> placed(segs.size(), -1), placed_inst(segs.size(), -1);
    std::vector<int32_t> row_leaves = bins[b].leaves;
    std::sort(row_leaves.begin(), row_leaves.end(),
              [&](int32_t x, int32_t y) { return leaves[x].rank < leaves[y].rank; });
    int32_t f = static_cast<int32_t>(fbase[b]), inst = static_cast<int32_t>(ibase[b]);
    for (int32_t li : row_leaves) {
      const Leaf& leaf = leaves[li];
      const int64_t rep_off = seq_offsets[leaf.rep()];
      int32_t prev = -1;
      for (int32_t s : leaf.path) {
        if (placed[s] < 0) {
          const int32_t L = segs[s].end - segs[s].start;
          placed[s] = f;
          placed_inst[s] = inst;
          inst_start[inst] = f;
          inst_len[inst] = L;
          inst_parent[inst] = prev >= 0 ? placed_inst[prev] : -1;
          // one segment = a chain: depths segs[s].start.., tokens copied,
          // each position's parent the one before it (the first one's: the
          // last position of the parent segment, or none at a root)
          std::iota(P.depth.begin() + f, P.depth.begin() + f + L, segs[s].start);
          std::memcpy(P.fwd_token.data() + f, tokens + rep_off + segs[s].start, sizeof(int32_t) * L);
          P.parent[f] = prev >= 0 ? placed[prev] + (segs[prev].end - 1 - segs[prev].start) : -1;
          std::iota(P.parent.begin() + f + 1, P.parent.begin() + f + L, f);
          std::fill(inst_of.begin() + f, inst_of.begin() + f + L, inst);
          f += L;
          ++inst;
        }
        prev = s;
      }
      for (int32_t m : leaf.members) {
        P.row_of_seq[m] = static_cast<int32_t>(b);
        const int64_t o = seq_offsets[m];
        for (int32_t s : leaf.path)
          for (int32_t p = segs[s].start; p < segs[s].end; ++p)
            P.token_index[o + p] = placed[s] + (p - segs[s].start);
      }
    }
  });
  // subtree ends, row by row (a parent always lies in its child's row, before it)
  P.subtree_end.resize(F);
  parallel_for(static_cast<int64_t>(nb), [&](int64_t b) {
    for (int64_t f = fbase[b]; f < fbase[b + 1]; ++f) P.subtree_end[f] = static_cast<int32_t>(f + 1);
    for (int64_t f = fbase[b + 1] - 1; f >= fbase[b]; --f) {
      const int32_t p = P.parent[f];
      if (p >= 0 && P.subtree_end[f] > P.subtree_end[p]) P.subtree_end[p] = P.subtree_end[f];
    }
  });
  // segment instances by tree level: the order in which a recurrent token
  // mixer threads its state through the tree ([ART] "Token-mixing layers",
  // GDN: one pass per tree depth, a child starting from its parent's final
  // state).  Level = number of ancestor instances (parents come first in
  // placement order); stable in placement order within a level.
  {
    const size_t ni = inst_start.size();
    std::vector<int32_t> level(ni);
    int32_t n_levels = 0;
    for (size_t i = 0; i < ni; ++i) {
      level[i] = inst_parent[i] < 0 ? 0 : level[static_cast<size_t>(inst_parent[i])] + 1;
      n_levels = std::max(n_levels, level[i] + 1);
    }
    P.seg_level_begin.assign(static_cast<size_t>(n_levels) + 1, 0);
    for (size_t i = 0; i < ni; ++i) ++P.seg_level_begin[static_cast<size_t>(level[i]) + 1];
    for (int32_t l = 0; l < n_levels; ++l) P.seg_level_begin[l + 1] += P.seg_level_begin[l];
    std::vector<int32_t> at(P.seg_level_begin.begin(), P.seg_level_begin.end() - 1), pos(ni);
    for (size_t i = 0; i < ni; ++i) pos[i] = at[static_cast<size_t>(level[i])]++;
    P.seg_start.resize(ni);
    P.seg_len.resize(ni);
    P.seg_parent.resize(ni);
    for (size_t i = 0; i < ni; ++i) {
      const size_t k = static_cast<size_t>(pos[i]);
      P.seg_start[k] = inst_start[i];
      P.seg_len[k] = inst_len[i];
      P.seg_parent[k] = inst_parent[i] < 0 ? -1 : pos[static_cast<size_t>(inst_parent[i])];
    }
    P.seg_off.resize(ni);
    for (int32_t l = 0; l < n_levels; ++l) {
      int32_t acc = 0;
      for (int32_t k = P.seg_level_begin[l]; k < P.seg_level_begin[l + 1]; ++k) {
        P.seg_off[static_cast<size_t>(k)] = acc;
        acc += P.seg_len[static_cast<size_t>(k)];
      }
    }
  }
  int64_t forks = 0;
  for (auto& s : segs) forks += (s.n_children >= 2);
  P.useful_pairs = 0;
  P.max_depth = 0;
  for (int64_t f = 0; f < F; ++f) {
    P.useful_pairs += P.depth[f] + 1;
    P.max_depth = std::max<int64_t>(P.max_depth, P.depth[f]);
  }
  P.packing_ratio = static_cast<double>(R) / static_cast<double>(F);
  P.row_fill_frac = static_cast<double>(F) / (static_cast<double>(P.n_rows) * static_cast<double>(C));
  P.fork_frac = static_cast<double>(forks) / static_cast<double>(segs.size());

  // ---- 5. work lists ------------------------------------------------------
  // Tiles sit on a per-row grid and read only their row, so every row builds
  // its own lists (begin offsets local to the row); they are then joined in
  // row order.
  struct RowLists {
    std::vector<int32_t> qt_q0, qt_nq, qt_kb_begin, kb, kt_k0, kt_nk, kt_qb_begin, qb;
    int64_t visited = 0;
  };
  std::vector<RowLists> lists(nb);
  parallel_for(static_cast<int64_t>(nb), [&](int64_t row) {
    RowLists& L = lists[static_cast<size_t>(row)];
    std::vector<int32_t> chain;
    std::vector<std::pair<int32_t, int32_t>> ivals;
    const int32_t rs = static_cast<int32_t>(fbase[row]);
    const int32_t re = static_cast<int32_t>(fbase[row + 1]);
    for (int32_t q0 = rs; q0 < re; q0 += kTile) {
      const int32_t q1 = std::min(q0 + kTile, re);
      L.qt_q0.push_back(q0);
      L.qt_nq.push_back(q1 - q0);
      L.qt_kb_begin.push_back(static_cast<int32_t>(L.kb.size() / 2));
      // ancestor chain of q0: proper ancestor instances, then q0's own prefix
      chain.clear();
      for (int32_t i = inst_parent[inst_of[q0]]; i >= 0; i = inst_parent[i]) chain.push_back(i);
      ivals.clear();
      for (size_t c = chain.size(); c-- > 0;) {
        const int32_t a0 = inst_start[chain[c]], e = a0 + inst_len[chain[c]];
        if (!ivals.empty() && ivals.back().second == a0) ivals.back().second = e;
        else ivals.push_back({a0, e});
      }
      const int32_t own = inst_start[inst_of[q0]];
      if (own < q0) {
        if (!ivals.empty() && ivals.back().second == own) ivals.back().second = q0;
        else ivals.push_back({own, q0});
      }
      ivals.push_back({q0, q1});   // the tile itself (causal + subtree mask)
      for (auto& iv : ivals) {
        for (int32_t k0 = iv.first; k0 < iv.second; k0 += kTile) {
          const int32_t nk = std::min(kTile, iv.second - k0);
          // full: the kernel may skip the mask -- all 128 loaded keys belong
          // to the block and every one is visible to every query of the tile.
          // Along an ancestor chain subtree ends do not increase, so the last
          // key of the block has the smallest one.
          const bool full = nk == kTile && (k0 + nk - 1 <= q0) && (P.subtree_end[k0 + nk - 1] >= q1);
          L.kb.push_back(k0);
          L.kb.push_back(nk | (full ? (1 << 16) : 0));
          L.visited += int64_t{kTile} * kTile;
        }
      }
    }
    for (int32_t k0 = rs; k0 < re; k0 += kTile) {
      const int32_t k1 = std::min(k0 + kTile, re);
      int32_t qend = 0, min_se = std::numeric_limits<int32_t>::max();
      for (int32_t j = k0; j < k1; ++j) {
        qend = std::max(qend, P.subtree_end[j]);
        min_se = std::min(min_se, P.subtree_end[j]);
      }
      L.kt_k0.push_back(k0);
      L.kt_nk.push_back(k1 - k0);
      L.kt_qb_begin.push_back(static_cast<int32_t>(L.qb.size() / 2));
      for (int32_t qs = k0; qs < qend; qs += kTile) {
        const int32_t qe = std::min(qs + kTile, qend);
        const bool full = (qe - qs == kTile) && (k1 - 1 <= qs) && (min_se >= qe);
        L.qb.push_back(qs);
        L.qb.push_back((qe - qs) | (full ? (1 << 16) : 0));
      }
    }
  });
  P.visited_pairs = 0;
  for (const RowLists& L : lists) {
    const size_t kb0 = P.kb.size() / 2, qb0 = P.qb.size() / 2;
    if (kb0 + L.kb.size() / 2 >= (size_t{1} << 31) || qb0 + L.qb.size() / 2 >= (size_t{1} << 31))
      return TPK_E_OVERFLOW;
    P.qt_q0.insert(P.qt_q0.end(), L.qt_q0.begin(), L.qt_q0.end());
    P.qt_nq.insert(P.qt_nq.end(), L.qt_nq.begin(), L.qt_nq.end());
    for (const int32_t x : L.qt_kb_begin) P.qt_kb_begin.push_back(static_cast<int32_t>(kb0) + x);
    P.kb.insert(P.kb.end(), L.kb.begin(), L.kb.end());
    P.kt_k0.insert(P.kt_k0.end(), L.kt_k0.begin(), L.kt_k0.end());
    P.kt_nk.insert(P.kt_nk.end(), L.kt_nk.begin(), L.kt_nk.end());
    for (const int32_t x : L.kt_qb_begin) P.kt_qb_begin.push_back(static_cast<int32_t>(qb0) + x);
    P.qb.insert(P.qb.end(), L.qb.begin(), L.qb.end());
    P.visited_pairs += L.visited;
  }
  if (P.kb.size() / 2 >= (size_t{1} << 31) || P.qb.size() / 2 >= (size_t{1} << 31)) return TPK_E_OVERFLOW;
  P.qt_kb_begin.push_back(static_cast<int32_t>(P.kb.size() / 2));
  P.kt_qb_begin.push_back(static_cast<int32_t>(P.qb.size() / 2));
  auto launch_order = [](const std::vector<int32_t>& begin) {
    const int32_t n = static_cast<int32_t>(begin.size()) - 1;
    const int32_t n_runs = (n + kOrderChunk - 1) / kOrderChunk;
    auto work = [&](int32_t t) { return begin[t + 1] - begin[t]; };
    std::vector<int64_t> run_work(n_runs, 0);
    for (int32_t t = 0; t < n; ++t) run_work[t / kOrderChunk] += work(t);
    std::vector<int32_t> runs(n_runs);
    std::iota(runs.begin(), runs.end(), 0);
    std::stable_sort(runs.begin(), runs.end(), [&](int32_t a, int32_t b) { return run_work[a] > run_work[b]; });
    std::vector<int32_t> o;
    o.reserve(n);
    for (int32_t r : runs) {
      const size_t first = o.size();
      for (int32_t t = r * kOrderChunk; t < std::min(n, (r + 1) * kOrderChunk); ++t) o.push_back(t);
      std::stable_sort(o.begin() + first, o.end(), [&](int32_t a, int32_t b) { return work(a) > work(b); });
    }
    return o;
  };
  P.qt_order = launch_order(P.qt_kb_begin);
  P.kt_order = launch_order(P.kt_qb_begin);

  // ---- raw tokens of each forwarded position (counting sort of token_index) --
  // A row's positions hold exactly the raw tokens of the row's sequences, so
  // each row sorts its own: its sequences in increasing index, their tokens
  // in order, keep every position's list ascending in raw index.  fwd_src,
  // the owner of a position, is the first of its list.
  {
    std::vector<int64_t> seq_begin(nb + 1, 0), raw_base(nb + 1, 0);
    for (int32_t q = 0; q < n_seqs; ++q) {
      ++seq_begin[P.row_of_seq[q] + 1];
      raw_base[P.row_of_seq[q] + 1] += len(q);
    }
    for (size_t b = 0; b < nb; ++b) {
      seq_begin[b + 1] += seq_begin[b];
      raw_base[b + 1] += raw_base[b];
    }
    std::vector<int32_t> row_seqs(static_cast<size_t>(n_seqs));
    {
      std::vector<int64_t> at(seq_begin.begin(), seq_begin.end() - 1);
      for (int32_t q = 0; q < n_seqs; ++q) row_seqs[at[P.row_of_seq[q]]++] = q;
    }
    P.fwd_raw_begin.resize(static_cast<size_t>(F) + 1);
    P.fwd_raw.resize(static_cast<size_t>(R));
    P.fwd_src.resize(static_cast<size_t>(F));
    parallel_for(static_cast<int64_t>(nb), [&](int64_t b) {
      const int64_t f0 = fbase[b], nf = fbase[b + 1] - fbase[b];
      std::vector<int64_t> at(static_cast<size_t>(nf) + 1, 0);
      for (int64_t k = seq_begin[b]; k < seq_begin[b + 1]; ++k) {
        const int32_t q = row_seqs[k];
        for (int64_t r = seq_offsets[q]; r < seq_offsets[q + 1]; ++r) ++at[P.token_index[r] - f0 + 1];
      }
      for (int64_t i = 0; i < nf; ++i) at[i + 1] += at[i];
      for (int64_t i = 0; i < nf; ++i) P.fwd_raw_begin[f0 + i] = static_cast<int32_t>(raw_base[b] + at[i]);
      for (int64_t k = seq_begin[b]; k < seq_begin[b + 1]; ++k) {
        const int32_t q = row_seqs[k];
        for (int64_t r = seq_offsets[q]; r < seq_offsets[q + 1]; ++r)
          P.fwd_raw[raw_base[b] + at[P.token_index[r] - f0]++] = static_cast<int32_t>(r);
      }
      for (int64_t i = 0; i < nf; ++i) P.fwd_src[f0 + i] = P.fwd_raw[P.fwd_raw_begin[f0 + i]];
    });
    P.fwd_raw_begin[F] = static_cast<int32_t>(R);
  }

  // ---- device image -------------------------------------------------------
  size_t off = 0;
  auto place = [&](size_t& field, size_t bytes) { field = off; off = align256(off + bytes); };
  place(P.off_depth, 4 * P.depth.size());
  place(P.off_token_index, 4 * P.token_index.size());
  place(P.off_subtree_end, 4 * P.subtree_end.size());
  place(P.off_parent, 4 * P.parent.size());
  place(P.off_fwd_raw_begin, 4 * P.fwd_raw_begin.size());
  place(P.off_fwd_raw, 4 * P.fwd_raw.size());
  place(P.off_qt_q0, 4 * P.qt_q0.size());
  place(P.off_qt_nq, 4 * P.qt_nq.size());
  place(P.off_qt_kb_begin, 4 * P.qt_kb_begin.size());
  place(P.off_kb, 4 * P.kb.size());
  place(P.off_qt_order, 4 * P.qt_order.size());
  place(P.off_kt_k0, 4 * P.kt_k0.size());
  place(P.off_kt_nk, 4 * P.kt_nk.size());
  place(P.off_kt_qb_begin, 4 * P.kt_qb_begin.size());
  place(P.off_qb, 4 * P.qb.size());
  place(P.off_kt_order, 4 * P.kt_order.size());
  place(P.off_seg_start, 4 * P.seg_start.size());
  place(P.off_seg_len, 4 * P.seg_len.size());
  place(P.off_seg_parent, 4 * P.seg_parent.size());
  place(P.off_seg_off, 4 * P.seg_off.size());
  // every byte is written once: the sections by copy, the padding after
  // each section (up to the next 256-byte boundary) with zeros; copied in
  // pieces of up to 4 MB on the host threads
  P.image.resize(off);
  struct Piece { size_t dst; const uint8_t* src; size_t bytes; };
  std::vector<Piece> pieces;
  auto put = [&](size_t field, const std::vector<int32_t>& v) {
    constexpr size_t kPiece = size_t{4} << 20;
    const auto* src = reinterpret_cast<const uint8_t*>(v.data());
    const size_t bytes = 4 * v.size();
    for (size_t b = 0; b < bytes; b += kPiece) pieces.push_back({field + b, src + b, std::min(kPiece, bytes - b)});
    const size_t end = field + bytes;
    pieces.push_back({end, nullptr, std::min(align256(end), off) - end});   // zeros
  };
  put(P.off_depth, P.depth);
  put(P.off_token_index, P.token_index);
  put(P.off_subtree_end, P.subtree_end);
  put(P.off_parent, P.parent);
  put(P.off_fwd_raw_begin, P.fwd_raw_begin);
  put(P.off_fwd_raw, P.fwd_raw);
  put(P.off_qt_q0, P.qt_q0);
  put(P.off_qt_nq, P.qt_nq);
  put(P.off_qt_kb_begin, P.qt_kb_begin);
  put(P.off_kb, P.kb);
  put(P.off_qt_order, P.qt_order);
  put(P.off_kt_k0, P.kt_k0);
  put(P.off_kt_nk, P.kt_nk);
  put(P.off_kt_qb_begin, P.kt_qb_begin);
  put(P.off_qb, P.qb);
  put(P.off_kt_order, P.kt_order);
  put(P.off_seg_start, P.seg_start);
  put(P.off_seg_len, P.seg_len);
  put(P.off_seg_parent, P.seg_parent);
  put(P.off_seg_off, P.seg_off);
  parallel_for(static_cast<int64_t>(pieces.size()), [&](int64_t i) {
    const Piece& pc = pieces[static_cast<size_t>(i)];
    if (pc.bytes == 0) return;
    if (pc.src) std::memcpy(P.image.data() + pc.dst, pc.src, pc.bytes);
    else std::memset(P.image.data() + pc.dst, 0, pc.bytes);
  });
  return TPK_OK;
}

}  // namespace tpk
