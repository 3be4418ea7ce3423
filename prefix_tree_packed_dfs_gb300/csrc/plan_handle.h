// The opaque handle behind `tpk_plan*`.
#pragma once
#include <cuda_runtime_api.h>

#include <mutex>

#include "planner.h"

struct tpk_plan {
  tpk::Plan p;
  // Page-locked copy of p.image, made by the first tpk_plan_upload so that
  // every upload is an asynchronous DMA instead of a copy staged through
  // pageable memory (which queues behind other host-to-device traffic).
  mutable void* pinned = nullptr;
  mutable size_t pinned_bytes = 0;
  mutable std::mutex pinned_mu;

  tpk_plan() = default;
  tpk_plan(const tpk_plan&) = delete;
  tpk_plan& operator=(const tpk_plan&) = delete;
  ~tpk_plan() {
    if (pinned) cudaFreeHost(pinned);
  }
};
