// profile.cu -- launch counter and per-stage CUDA-event timing of the forward.
#include <atomic>
#include <mutex>
#include <vector>

#include "mlr_profile.cuh"

namespace mlr {
namespace {

std::atomic<uint64_t> g_launches{0};
std::atomic<uint64_t> g_wait_ns{kWaitLimitNs};
std::atomic<int> g_deterministic{1};  // measured no slower than the atomic combine
std::mutex g_mu;
bool g_on = false;
int g_max_calls = 0, g_calls = 0;
std::vector<cudaEvent_t> g_events;  // [max_calls][kProfStages + 1]
constexpr uint32_t kAllStages = (1u << kProfStages) - 1;
uint32_t g_select = kAllStages;  // stages that the next begin() times
uint32_t g_mask = kAllStages;    // stages timed by the current recording

// Boundary b (0 = call start, b = s + 1 after stage s) is recorded when a
// selected stage starts or ends there.
bool boundary_needed(int b) {
  return ((b < kProfStages && ((g_mask >> b) & 1)) || (b > 0 && ((g_mask >> (b - 1)) & 1)));
}

const char* kStageNames[kProfStages] = {"align_plan", "gather", "shrink_gate_up", "gate_up",
                                        "shrink_down", "down", "convert"};

}  // namespace

void note_launch(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

uint64_t wait_limit_ns() { return g_wait_ns.load(std::memory_order_relaxed); }

bool combine_deterministic() { return g_deterministic.load(std::memory_order_relaxed) != 0; }

int prof_call_begin(cudaStream_t stream) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_on || g_calls >= g_max_calls) return -1;
  const int slot = g_calls++;
  if (boundary_needed(0)) cudaEventRecord(g_events[(size_t)slot * (kProfStages + 1)], stream);
  return slot;
}

void prof_mark(int slot, int stage, cudaStream_t stream) {
  if (slot < 0 || !boundary_needed(stage + 1)) return;
  cudaEventRecord(g_events[(size_t)slot * (kProfStages + 1) + stage + 1], stream);
}

}  // namespace mlr

extern "C" int moe_lora_profile_begin(int32_t max_calls) {
  using namespace mlr;
  if (max_calls < 1 || max_calls > 4096) return MLR_ERR_INVALID;
  std::lock_guard<std::mutex> lk(g_mu);
  const size_t need = (size_t)max_calls * (kProfStages + 1);
  while (g_events.size() < need) {
    cudaEvent_t e;
    if (cudaEventCreate(&e) != cudaSuccess) return MLR_ERR_CUDA;
    g_events.push_back(e);
  }
  g_max_calls = max_calls;
  g_calls = 0;
  g_mask = g_select;
  g_on = true;
  return MLR_OK;
}

extern "C" int moe_lora_profile_stages(uint32_t mask) {
  using namespace mlr;
  if (mask == 0 || (mask & ~kAllStages) != 0) return MLR_ERR_INVALID;
  std::lock_guard<std::mutex> lk(g_mu);
  g_select = mask;
  return MLR_OK;
}

extern "C" int moe_lora_profile_end(double* stage_ms, int32_t max_stages, int32_t* n_stages,
                                    int32_t* n_calls) {
  using namespace mlr;
  std::lock_guard<std::mutex> lk(g_mu);
  g_on = false;
  if (n_stages) *n_stages = kProfStages;
  if (n_calls) *n_calls = g_calls;
  if (stage_ms == nullptr) return MLR_OK;
  for (int s = 0; s < max_stages && s < kProfStages; ++s) stage_ms[s] = 0.0;
  int last = 0;  // the last boundary recorded in every call
  for (int b = 0; b <= kProfStages; ++b)
    if (boundary_needed(b)) last = b;
  for (int c = 0; c < g_calls; ++c) {
    cudaEvent_t* ev = &g_events[(size_t)c * (kProfStages + 1)];
    if (cudaEventSynchronize(ev[last]) != cudaSuccess) return MLR_ERR_CUDA;
    for (int s = 0; s < max_stages && s < kProfStages; ++s) {
      if (((g_mask >> s) & 1) == 0) continue;
      float ms = 0.f;
      if (cudaEventElapsedTime(&ms, ev[s], ev[s + 1]) != cudaSuccess) return MLR_ERR_CUDA;
      stage_ms[s] += ms;
    }
  }
  return MLR_OK;
}

extern "C" const char* moe_lora_profile_stage_name(int32_t stage) {
  return (stage >= 0 && stage < mlr::kProfStages) ? mlr::kStageNames[stage] : nullptr;
}

extern "C" uint64_t moe_lora_launch_count(void) { return mlr::g_launches.load(); }

extern "C" int moe_lora_set_wait_limit_ns(uint64_t ns) {
  if (ns > mlr::kMaxWaitLimitNs) return MLR_ERR_INVALID;
  mlr::g_wait_ns.store(ns == 0 ? 1 : ns, std::memory_order_relaxed);
  return MLR_OK;
}

extern "C" uint64_t moe_lora_wait_limit_ns(void) { return mlr::wait_limit_ns(); }

extern "C" int moe_lora_set_deterministic(int32_t on) {
  if (on != 0 && on != 1) return MLR_ERR_INVALID;
  mlr::g_deterministic.store(on, std::memory_order_relaxed);
  return MLR_OK;
}

extern "C" int32_t moe_lora_deterministic(void) { return mlr::combine_deterministic() ? 1 : 0; }
