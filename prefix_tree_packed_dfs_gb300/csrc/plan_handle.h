// The opaque handle behind `tpk_plan*`.
#pragma once
#include "planner.h"

struct tpk_plan {
  tpk::Plan p;
};
