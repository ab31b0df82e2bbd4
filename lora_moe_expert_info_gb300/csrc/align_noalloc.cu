// align_noalloc.cu -- moe_lora_align_noalloc: the (expert, adapter) align for
// callers that may not allocate device memory.
//
// Some callers cannot hand this library a workspace: a serving engine that
// reserves all of the GPU's memory for its own pools at start-up and forbids any
// later allocation, code on a latency-critical path where cudaMalloc/cudaFree
// could synchronise the device, or a layer that is simply given no allocator.
// For them the align's scratch (per-chunk bucket counts and bucket offsets)
// lives in a fixed array that is part of this library's device image: every
// GPU that loads the library holds kNoAllocScratchBytes for it until the
// process exits.  The entry point itself never calls cudaMalloc, cudaFree or
// any allocating routine.
#include <mutex>

#include "mlr_align.cuh"

namespace mlr {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;  // 4 MiB
constexpr int kMaxDevices = 64;

std::mutex g_mu;
void* g_scratch_dev_ptr[kMaxDevices] = {};

}  // namespace
}  // namespace mlr

// The shared scratch.  In host code this name is only a stand-in for the
// device array, never a device address: the address is looked up per device.
static __device__ __align__(256) unsigned char g_align_scratch[mlr::kNoAllocScratchBytes];

namespace mlr {
namespace {

// Device address of the scratch array on the current device, looked up once
// per device (the lookup may load this library's module onto that device).
// The cache is keyed by device ordinal: it assumes the device's primary
// context (the one the CUDA runtime uses) for the life of the process.  After
// cudaDeviceReset, or under another driver-API context made current, the
// cached address would be stale, so callers doing either must not use this
// entry point afterwards.
int scratch_for_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    (void)cudaGetLastError();
    return MLR_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_scratch_dev_ptr[dev] == nullptr) {
    void* p = nullptr;
    const cudaError_t err = cudaGetSymbolAddress(&p, g_align_scratch);
    if (err != cudaSuccess || p == nullptr) {
      (void)cudaGetLastError();
      return MLR_ERR_CUDA;
    }
    g_scratch_dev_ptr[dev] = p;
  }
  *out = g_scratch_dev_ptr[dev];
  return MLR_OK;
}

}  // namespace
}  // namespace mlr

extern "C" int moe_lora_align_noalloc(const int32_t* topk_ids, const int32_t* token_lora_mapping,
                                      int32_t num_tokens, int32_t topk, int32_t num_experts,
                                      int32_t num_loras, int32_t block_size,
                                      int32_t* sorted_token_ids, int32_t* block_expert_ids,
                                      int32_t* block_lora_ids, int32_t* num_tokens_post_pad,
                                      int64_t capacity, int32_t* d_status, void* stream) {
  using namespace mlr;
  const AlignPlan pl = align_plan(num_tokens, topk, num_experts, num_loras, block_size);
  if (!pl.ok) {
    if (num_tokens < 0 || topk < 1 || num_experts < 1 || num_loras < 0 || block_size < 1)
      return MLR_ERR_INVALID;
    return MLR_ERR_UNSUPPORTED;
  }
  if (num_tokens_post_pad == nullptr || capacity < 0) return MLR_ERR_INVALID;
  if (pl.P > 0 && (topk_ids == nullptr || token_lora_mapping == nullptr)) return MLR_ERR_INVALID;
  if (capacity > 0 && (sorted_token_ids == nullptr || block_expert_ids == nullptr ||
                       block_lora_ids == nullptr))
    return MLR_ERR_INVALID;
  // Sizes whose scratch does not fit the fixed array are refused up front.
  if ((size_t)pl.ws_bytes > kNoAllocScratchBytes) return MLR_ERR_CAPACITY;
  void* scratch = nullptr;
  const int rc = scratch_for_current_device(&scratch);
  if (rc != MLR_OK) return rc;
  // Every scratch word the four align launches read is written by an earlier
  // launch of the same call, so nothing has to be cleared between calls.
  return align_launch(pl, topk_ids, token_lora_mapping, topk, num_experts, num_loras, block_size,
                      sorted_token_ids, block_expert_ids, block_lora_ids, num_tokens_post_pad,
                      capacity, scratch, d_status, static_cast<cudaStream_t>(stream));
}
