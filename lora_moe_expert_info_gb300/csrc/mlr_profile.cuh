// mlr_profile.cuh -- launch counting and optional per-stage event recording.
#pragma once
#include "mlr_common.cuh"

namespace mlr {

constexpr int kProfStages = 7;  // align, plan + x gather, shrink_gu, gate_up, shrink_d, down, convert

void note_launch(int n = 1);
// Per forward call: returns a slot (>= 0) while recording is on, else -1.
int prof_call_begin(cudaStream_t stream);
// Records the boundary after `stage` (0-based) for the call slot.
void prof_mark(int slot, int stage, cudaStream_t stream);
// Give-up limit of the GEMM kernels' pipeline waits for the next launches
// (moe_lora_set_wait_limit_ns; kWaitLimitNs by default).
uint64_t wait_limit_ns();
// Top-k combine of the MoE forward for the next calls: fp32 reductions into
// y_acc (false) or per-pair rows summed in a fixed order (true).
bool combine_deterministic();

}  // namespace mlr
