// profile.cu -- optional per-kernel timing of the library's own launches.
//
// When enabled, every kernel launch (or, with boost_profile_only, every launch of one
// kernel) is bracketed by two CUDA events recorded on the launch's stream, and the launch's algorithmic work (flops and bytes, from the
// shapes) is accumulated per kernel. Reading the counters synchronises the pending
// events. Disabled (the default), a launch pays one relaxed atomic load. While the
// stream is being captured into a CUDA graph the events become event-record nodes of
// the graph (recorded when the graph runs), so a graph captured with timing enabled
// and launched once yields one sample per captured launch.
#include "profile.h"

#include <atomic>
#include <mutex>
#include <vector>

namespace boost_gb300 {

namespace {

const char* const kNames[K_COUNT] = {
    "rmsnorm_stats", "fold_gamma",     "gemm_down_act",  "gemm_up",
    "gemm_dual",     "gemm_wgrad_B",   "gemm_wgrad_A",   "gemm_dx",
    "splitk_sum",    "splitk_finalize_dA", "dgamma_reduce", "swiglu_fwd",
    "swiglu_bwd",    "add",            "wait_probe",    "gemm_dx_swiglu",
    "gemm_up_swiglu", "gemm_down_partials", "btp_exchange_reduce", "rmsnorm_stats_fold"};

struct Pending {
  int id;
  cudaEvent_t e0, e1;
  double flops, bytes;
  int kernels;
};

struct Totals {
  int64_t launches = 0, kernels = 0;
  double ms = 0.0, flops = 0.0, bytes = 0.0;
};

std::atomic<int> g_enabled{0};
std::atomic<int> g_only{-1};   // the one kernel id timed, or -1 for all
std::mutex g_mu;
std::vector<Pending> g_pending;
std::vector<cudaEvent_t> g_pool;
Totals g_tot[K_COUNT];
thread_local ProfScope* t_open = nullptr;

cudaEvent_t take_event() {
  if (!g_pool.empty()) {
    cudaEvent_t e = g_pool.back();
    g_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return e;
}

void drain_locked() {
  for (Pending& p : g_pending) {
    float ms = 0.0f;
    if (cudaEventSynchronize(p.e1) == cudaSuccess &&
        cudaEventElapsedTime(&ms, p.e0, p.e1) == cudaSuccess) {
      Totals& t = g_tot[p.id];
      t.launches += 1;
      t.kernels += p.kernels;
      t.ms += ms;
      t.flops += p.flops;
      t.bytes += p.bytes;
    } else {
      cudaGetLastError();
    }
    g_pool.push_back(p.e0);
    g_pool.push_back(p.e1);
  }
  g_pending.clear();
}

void record(cudaEvent_t e, cudaStream_t s) {
  cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &st) == cudaSuccess && st == cudaStreamCaptureStatusActive)
    cudaEventRecordWithFlags(e, s, cudaEventRecordExternal);
  else
    cudaEventRecord(e, s);
}

}  // namespace

ProfScope::ProfScope(cudaStream_t s, int id, double flops, double bytes)
    : stream_(s), id_(id), flops_(flops), bytes_(bytes) {
  if (g_enabled.load(std::memory_order_relaxed) == 0) return;
  const int only = g_only.load(std::memory_order_relaxed);
  if (only >= 0 && only != id) return;
  std::lock_guard<std::mutex> lk(g_mu);
  e0_ = take_event();
  e1_ = take_event();
  if (e0_ && e1_) {
    record(e0_, stream_);
    active_ = true;
    outer_ = t_open;
    t_open = this;
  }
}

ProfScope::~ProfScope() {
  if (!active_) return;
  t_open = outer_;
  std::lock_guard<std::mutex> lk(g_mu);
  record(e1_, stream_);
  g_pending.push_back(Pending{id_, e0_, e1_, flops_, bytes_, kernels_});
}

void prof_note_kernels(int extra) {
  if (t_open != nullptr) t_open->kernels_ += extra;
}

}  // namespace boost_gb300

using namespace boost_gb300;

extern "C" {

boost_status boost_profile_enable(int on) {
  std::lock_guard<std::mutex> lk(g_mu);
  drain_locked();
  if (on) {
    for (auto& t : g_tot) t = Totals{};
  }
  g_enabled.store(on ? 1 : 0);
  return BOOST_OK;
}

boost_status boost_profile_only(int id) {
  if (id < -1 || id >= K_COUNT) return BOOST_ERR_INVALID_ARG;
  g_only.store(id);
  return BOOST_OK;
}

int boost_profile_kernel_count(void) { return K_COUNT; }

boost_status boost_profile_read_kernels(int id, int64_t* kernels) {
  if (id < 0 || id >= K_COUNT || kernels == nullptr) return BOOST_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_mu);
  drain_locked();
  *kernels = g_tot[id].kernels;
  return BOOST_OK;
}

boost_status boost_profile_read(int id, const char** name, int64_t* launches, double* total_ms,
                                double* total_flops, double* total_bytes) {
  if (id < 0 || id >= K_COUNT) return BOOST_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_mu);
  drain_locked();
  const Totals& t = g_tot[id];
  if (name) *name = kNames[id];
  if (launches) *launches = t.launches;
  if (total_ms) *total_ms = t.ms;
  if (total_flops) *total_flops = t.flops;
  if (total_bytes) *total_bytes = t.bytes;
  return BOOST_OK;
}

}  // extern "C"
