// Exposes the schedule formulas of the kernels' schedule.h to the CPU tests.
#include <cstdint>

#include "schedule.h"

extern "C" int32_t sched_worker_begin(int32_t c, int32_t total, int32_t grid) {
  return mla::worker_begin(c, total, grid);
}
extern "C" int32_t sched_worker_of_tile(int32_t t, int32_t total, int32_t grid) {
  return mla::worker_of_tile(t, total, grid);
}
