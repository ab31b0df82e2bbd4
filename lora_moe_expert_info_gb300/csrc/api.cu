// api.cu -- version and status-code text of the C ABI.
#include "mlr_common.cuh"

extern "C" const char* moe_lora_version(void) { return "moe_lora 0.1.0 (sm_103a)"; }

extern "C" const char* moe_lora_status_string(int code) {
  switch (code) {
    case MLR_OK: return "ok";
    case MLR_ERR_INVALID: return "invalid argument";
    case MLR_ERR_UNDERCOVERED: return "launch under-covers tokens (bs * max_len < num_tokens)";
    case MLR_ERR_INDEX: return "id out of range";
    case MLR_ERR_CAPACITY: return "capacity or workspace too small";
    case MLR_ERR_CUDA: return "CUDA launch or driver call failed";
    case MLR_ERR_TIMEOUT: return "device wait timed out";
    case MLR_ERR_UNSUPPORTED: return "shape not supported by the kernels";
    default: return "unknown status";
  }
}
