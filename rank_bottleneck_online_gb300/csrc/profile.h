// profile.h -- per-kernel launch timing of the library (see profile.cu).
#pragma once

#include <cuda_runtime.h>

#include "boost_block.h"

namespace boost_gb300 {

enum KernelId : int {
  K_STATS = 0,
  K_FOLD,
  K_DOWN,
  K_UP,
  K_DUAL,
  K_WGRAD_B,
  K_WGRAD_A,
  K_DX,
  K_SPLITK_SUM,
  K_FINALIZE_DA,
  K_DGAMMA,
  K_SWIGLU_FWD,
  K_SWIGLU_BWD,
  K_ADD,
  K_PROBE,
  K_DX_GLU,
  K_UP_GLU,
  K_BTP_PARTIAL,
  K_BTP_REDUCE,
  K_STATS_FOLD,
  K_COUNT
};

// Brackets one operation with events on `s` when profiling is enabled; `flops` and
// `bytes` are the operation's algorithmic work. An operation is one kernel launch
// unless the code inside the scope reports more with prof_note_kernels.
class ProfScope {
 public:
  ProfScope(cudaStream_t s, int id, double flops, double bytes);
  ~ProfScope();
  ProfScope(const ProfScope&) = delete;
  ProfScope& operator=(const ProfScope&) = delete;

 private:
  cudaStream_t stream_;
  int id_;
  double flops_, bytes_;
  cudaEvent_t e0_ = nullptr, e1_ = nullptr;
  bool active_ = false;
  int kernels_ = 1;
  ProfScope* outer_ = nullptr;
  friend void prof_note_kernels(int extra);
};

// Adds `extra` kernel launches to the innermost open scope of this thread (an
// operation split over several concurrent launches).
void prof_note_kernels(int extra);

}  // namespace boost_gb300
