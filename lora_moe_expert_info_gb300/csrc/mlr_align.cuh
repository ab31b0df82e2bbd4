// mlr_align.cuh -- internal interface of the (expert, adapter) align, shared by
// moe_lora_align and the forward (which runs the align with block 16).
#pragma once
#include "mlr_common.cuh"

namespace mlr {

constexpr int64_t kMaxAlignBuckets = 40960;  // E*(L+1): histogram + chunk fit in shared memory
constexpr int kMaxAlignBlock = 4096;

struct AlignPlan {
  bool ok;
  int64_t P;          // pairs
  int NB;             // buckets E*(L+1)
  int chunk;          // pairs per chunk
  int G;              // chunks
  int64_t capacity;   // padded-length bound
  int64_t cnt_off, btotal_off, bstart_off, ws_bytes;  // workspace layout (bytes)
};

AlignPlan align_plan(int32_t num_tokens, int32_t topk, int32_t num_experts, int32_t num_loras,
                     int32_t block_size);

// Enqueues the four align launches.  Workspace holds cnt[G][NB], btotal[NB]
// (pairs per bucket) and bstart[NB+1] (padded bucket starts; bstart[NB] = total).
int align_launch(const AlignPlan& pl, const int32_t* topk_ids, const int32_t* mapping, int topk,
                 int E, int L, int block_size, int32_t* sorted_ids, int32_t* block_expert,
                 int32_t* block_lora, int32_t* num_post_pad, int64_t capacity, void* workspace,
                 int32_t* d_status, cudaStream_t stream);

}  // namespace mlr
