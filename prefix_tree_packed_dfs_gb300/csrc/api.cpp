// C ABI: planner entry points, device image upload, status strings.
#include <cuda_runtime_api.h>

#include <algorithm>
#include <cstring>
#include <mutex>
#include <new>
#include <numeric>
#include <utility>
#include <vector>

#include "plan_handle.h"
#include "tpk.h"

namespace {
// Page-locked buffers of destroyed plans, kept for the next plans' uploads:
// allocating and freeing page-locked memory costs far more than the copy, and
// callers that plan every step would pay it every step.  At most two are kept.
std::mutex g_pinned_mu;
std::vector<std::pair<void*, size_t>> g_pinned_free;
constexpr size_t kMaxFreePinned = 2;

void* take_pinned(size_t bytes, size_t* got) {
  std::lock_guard<std::mutex> lock(g_pinned_mu);
  size_t best = g_pinned_free.size();
  for (size_t i = 0; i < g_pinned_free.size(); ++i)
    if (g_pinned_free[i].second >= bytes && (best == g_pinned_free.size() || g_pinned_free[i].second < g_pinned_free[best].second))
      best = i;
  if (best == g_pinned_free.size()) return nullptr;
  void* p = g_pinned_free[best].first;
  *got = g_pinned_free[best].second;
  g_pinned_free.erase(g_pinned_free.begin() + static_cast<std::ptrdiff_t>(best));
  return p;
}

void give_pinned(void* p, size_t bytes) {
  void* drop = p;
  {
    std::lock_guard<std::mutex> lock(g_pinned_mu);
    if (g_pinned_free.size() < kMaxFreePinned) {
      g_pinned_free.push_back({p, bytes});
      return;
    }
    // full: keep the larger buffers
    size_t smallest = 0;
    for (size_t i = 1; i < g_pinned_free.size(); ++i)
      if (g_pinned_free[i].second < g_pinned_free[smallest].second) smallest = i;
    if (g_pinned_free[smallest].second < bytes) {
      drop = g_pinned_free[smallest].first;
      g_pinned_free[smallest] = {p, bytes};
    }
  }
  cudaFreeHost(drop);
}

template <typename T, typename U>
void copy_out(T* dst, const std::vector<U>& v) {
  if (dst)
    for (size_t i = 0; i < v.size(); ++i) dst[i] = static_cast<T>(v[i]);
}
// The arrays of the last destroyed plan, kept for the next build: a training
// loop plans one batch per step, and building into memory that is already
// mapped skips the page faults of fresh allocations (most of what the
// planner spends on a large batch after its parallel passes).  At most one
// plan's storage is kept.
std::mutex g_plan_mu;
tpk::Plan g_plan_free;
bool g_plan_free_held = false;

void take_plan_storage(tpk::Plan* p) {
  std::lock_guard<std::mutex> lock(g_plan_mu);
  if (!g_plan_free_held) return;
  std::swap(*p, g_plan_free);
  g_plan_free_held = false;
}

void give_plan_storage(tpk::Plan* p) {
  std::lock_guard<std::mutex> lock(g_plan_mu);
  std::swap(*p, g_plan_free);   // the previous spare, if any, is freed with the handle
  g_plan_free_held = true;
}

}  // namespace

extern "C" {

int tpk_plan_build(const int32_t* tokens, const int64_t* seq_offsets, int32_t n_seqs,
                   const uint8_t* trained, const int32_t* group_ids,
                   const tpk_plan_opts* opts, tpk_plan** out) {
  if (!out) return TPK_E_ARG;
  *out = nullptr;
  tpk::PlanOptions o;
  if (opts) {
    o.row_capacity = opts->row_capacity;
    o.min_shared = opts->min_shared;
    o.placement = opts->placement;
  }
  tpk_plan* h = new (std::nothrow) tpk_plan();
  if (!h) return TPK_E_ARG;
  take_plan_storage(&h->p);
  int st;
  // nothing thrown inside the planner (out of host memory, a worker thread
  // that could not be created, ...) may cross the C ABI
  try {
    st = tpk::build_plan(tokens, seq_offsets, n_seqs, trained, group_ids, o, &h->p);
  } catch (const std::bad_alloc&) {
    st = TPK_E_HOST;
  } catch (...) {
    st = TPK_E_HOST;
  }
  if (st != TPK_OK) {
    delete h;
    return st;
  }
  *out = h;
  return TPK_OK;
}

int tpk_plan_info_get(const tpk_plan* plan, tpk_plan_info* out) {
  if (!plan || !out) return TPK_E_ARG;
  const tpk::Plan& P = plan->p;
  out->n_seqs = P.n_seqs;
  out->n_rows = P.n_rows;
  out->n_fwd = P.F;
  out->n_raw = P.R;
  out->n_segments = P.n_segments;
  out->n_leaves = P.n_leaves;
  out->n_qtiles = static_cast<int64_t>(P.qt_q0.size());
  out->n_kblocks = static_cast<int64_t>(P.kb.size() / 2);
  out->n_ktiles = static_cast<int64_t>(P.kt_k0.size());
  out->n_qblocks = static_cast<int64_t>(P.qb.size() / 2);
  out->useful_pairs = P.useful_pairs;
  out->visited_pairs = P.visited_pairs;
  out->max_depth = P.max_depth;
  out->packing_ratio = P.packing_ratio;
  out->row_fill_frac = P.row_fill_frac;
  out->fork_frac = P.fork_frac;
  out->n_seg_instances = static_cast<int64_t>(P.seg_start.size());
  out->n_seg_levels = P.seg_level_begin.empty() ? 0 : static_cast<int64_t>(P.seg_level_begin.size()) - 1;
  return TPK_OK;
}

int tpk_plan_export(const tpk_plan* plan, int64_t* row_offsets, int64_t* row_loads,
                    int32_t* row_of_seq, int32_t* fwd_token, int32_t* fwd_src,
                    int32_t* parent, int32_t* depth, int32_t* token_index,
                    int32_t* subtree_end) {
  if (!plan) return TPK_E_ARG;
  const tpk::Plan& P = plan->p;
  copy_out(row_offsets, P.row_offsets);
  copy_out(row_loads, P.row_loads);
  copy_out(row_of_seq, P.row_of_seq);
  copy_out(fwd_token, P.fwd_token);
  copy_out(fwd_src, P.fwd_src);
  copy_out(parent, P.parent);
  copy_out(depth, P.depth);
  copy_out(token_index, P.token_index);
  copy_out(subtree_end, P.subtree_end);
  return TPK_OK;
}

int tpk_plan_worklists(const tpk_plan* plan, int32_t* qt_q0, int32_t* qt_nq,
                       int32_t* qt_kb_begin, int32_t* kb, int32_t* qt_order,
                       int32_t* kt_k0, int32_t* kt_nk, int32_t* kt_qb_begin,
                       int32_t* qb, int32_t* kt_order) {
  if (!plan) return TPK_E_ARG;
  const tpk::Plan& P = plan->p;
  copy_out(qt_q0, P.qt_q0);
  copy_out(qt_nq, P.qt_nq);
  copy_out(qt_kb_begin, P.qt_kb_begin);
  copy_out(kb, P.kb);
  copy_out(qt_order, P.qt_order);
  copy_out(kt_k0, P.kt_k0);
  copy_out(kt_nk, P.kt_nk);
  copy_out(kt_qb_begin, P.kt_qb_begin);
  copy_out(qb, P.qb);
  copy_out(kt_order, P.kt_order);
  return TPK_OK;
}

int tpk_plan_raw_of_forwarded(const tpk_plan* plan, int32_t* fwd_raw_begin, int32_t* fwd_raw) {
  if (!plan) return TPK_E_ARG;
  copy_out(fwd_raw_begin, plan->p.fwd_raw_begin);
  copy_out(fwd_raw, plan->p.fwd_raw);
  return TPK_OK;
}

int tpk_plan_segments(const tpk_plan* plan, int32_t* level_begin, int32_t* seg_start, int32_t* seg_len,
                      int32_t* seg_parent) {
  if (!plan) return TPK_E_ARG;
  copy_out(level_begin, plan->p.seg_level_begin);
  copy_out(seg_start, plan->p.seg_start);
  copy_out(seg_len, plan->p.seg_len);
  copy_out(seg_parent, plan->p.seg_parent);
  return TPK_OK;
}

int tpk_plan_shard_rows(const tpk_plan* plan, int32_t world, int32_t* rank_of_row, int64_t* rank_pairs) {
  if (!plan || world <= 0 || !rank_of_row) return TPK_E_ARG;
  const tpk::Plan& P = plan->p;
  const size_t rows = P.row_loads.size();
  // a row's work: its useful (query, key) pairs, sum of depth + 1 over its positions
  std::vector<int64_t> pairs(rows, 0);
  for (size_t r = 0; r < rows; ++r)
    for (int64_t f = P.row_offsets[r]; f < P.row_offsets[r + 1]; ++f) pairs[r] += static_cast<int64_t>(P.depth[f]) + 1;
  // longest processing time first: heaviest row to the least loaded rank
  // (ties: the lower row, the lower rank), so the assignment is reproducible
  std::vector<int32_t> order(rows);
  std::iota(order.begin(), order.end(), 0);
  std::stable_sort(order.begin(), order.end(), [&](int32_t a, int32_t b) { return pairs[a] > pairs[b]; });
  std::vector<int64_t> load(static_cast<size_t>(world), 0);
  for (const int32_t r : order) {
    size_t k = 0;
    for (size_t j = 1; j < load.size(); ++j)
      if (load[j] < load[k]) k = j;
    rank_of_row[r] = static_cast<int32_t>(k);
    load[k] += pairs[r];
  }
  if (rank_pairs) std::copy(load.begin(), load.end(), rank_pairs);
  return TPK_OK;
}

size_t tpk_plan_device_bytes(const tpk_plan* plan) { return plan ? plan->p.image.size() : 0; }

int tpk_plan_field_offset(const tpk_plan* plan, int32_t field, size_t* offset) {
  if (!plan || !offset) return TPK_E_ARG;
  switch (field) {
    case TPK_FIELD_DEPTH: *offset = plan->p.off_depth; return TPK_OK;
    case TPK_FIELD_TOKEN_INDEX: *offset = plan->p.off_token_index; return TPK_OK;
    case TPK_FIELD_SUBTREE_END: *offset = plan->p.off_subtree_end; return TPK_OK;
    case TPK_FIELD_PARENT: *offset = plan->p.off_parent; return TPK_OK;
    case TPK_FIELD_FWD_RAW_BEGIN: *offset = plan->p.off_fwd_raw_begin; return TPK_OK;
    case TPK_FIELD_FWD_RAW: *offset = plan->p.off_fwd_raw; return TPK_OK;
    case TPK_FIELD_SEG_START: *offset = plan->p.off_seg_start; return TPK_OK;
    case TPK_FIELD_SEG_LEN: *offset = plan->p.off_seg_len; return TPK_OK;
    case TPK_FIELD_SEG_PARENT: *offset = plan->p.off_seg_parent; return TPK_OK;
    case TPK_FIELD_SEG_OFF: *offset = plan->p.off_seg_off; return TPK_OK;
    default: return TPK_E_ARG;
  }
}

int tpk_plan_upload(const tpk_plan* plan, void* dev_image, void* stream) {
  if (!plan || !dev_image) return TPK_E_ARG;
  if (reinterpret_cast<uintptr_t>(dev_image) % 256) return TPK_E_ARG;
  const auto& img = plan->p.image;
  if (img.empty()) return TPK_OK;
  const void* src = img.data();
  {
    std::lock_guard<std::mutex> lock(plan->pinned_mu);
    if (!plan->pinned) {
      size_t got = 0;
      void* h = take_pinned(img.size(), &got);
      if (!h) {
        if (cudaMallocHost(&h, img.size()) == cudaSuccess) {
          got = img.size();
        } else {
          h = nullptr;
          (void)cudaGetLastError();   // no page-locked memory: copy from the pageable image
        }
      }
      if (h) {
        std::memcpy(h, img.data(), img.size());
        plan->pinned = h;
        plan->pinned_bytes = got;
      }
    }
    if (plan->pinned) src = plan->pinned;
  }
  cudaError_t e = cudaMemcpyAsync(dev_image, src, img.size(), cudaMemcpyHostToDevice,
                                  static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? TPK_OK : TPK_E_CUDA;
}

void tpk_plan_destroy(tpk_plan* plan) {
  if (!plan) return;
  if (plan->pinned) {
    give_pinned(plan->pinned, plan->pinned_bytes);
    plan->pinned = nullptr;
  }
  give_plan_storage(&plan->p);
  delete plan;
}

const char* tpk_status_string(int status) {
  switch (status) {
    case TPK_OK: return "ok";
    case TPK_E_ARG: return "invalid argument";
    case TPK_E_SEQ_TOO_LONG: return "a sequence is longer than the row capacity";
    case TPK_E_OVERFLOW: return "size does not fit the int32 layout";
    case TPK_E_UNSUPPORTED: return "unsupported shape or device (needs sm_103, head_dim 64/128, Hq % Hkv == 0)";
    case TPK_E_CUDA: return "CUDA call failed";
    case TPK_E_TIMEOUT: return "a device wait gave up";
    case TPK_E_WORKSPACE: return "workspace missing or too small";
    case TPK_E_SCRATCH_LIMIT: return "problem too large for the no-allocation backward's 32 MiB static scratch (Hq * F > 8388608)";
    case TPK_E_HOST: return "host-side failure inside the planner (out of host memory or another C++ exception)";
    default: return "unknown status";
  }
}

const char* tpk_version(void) { return "tpk 0.1 (sm_103a)"; }

}  // extern "C"
