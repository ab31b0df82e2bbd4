// tp_lora.cu -- column-parallel LoRA B of a fused q/k/v projection: the rows of
// the stacked B (outputs q, then k, then v) that one tensor-parallel rank
// holds.  Host code only.
//
// sglang PR #24420 page ("qkv_proj LoRA B sizing under KV-head replication"),
// 关键源码片段: mem_pool.py `_column_parallel_lora_b_per_rank_dim` and
// layers.py `slice_lora_b_weights`.  While the TP size does not exceed the
// number of KV heads, each rank takes an even 1/tp of the q rows and of the k
// and v rows.  Beyond it, each KV head is replicated over tp / num_kv_heads
// ranks: a rank takes its 1/tp of the q rows and one whole head (head_dim
// rows) of k and of v, the head of index rank / replicas.
#include <cstdint>

#include "moe_lora.h"

extern "C" int lora_tp_qkv_b_rows(int32_t num_heads, int32_t num_kv_heads, int32_t head_dim, int32_t tp_size,
                                  int32_t tp_rank, int32_t* ranges, int32_t* per_rank_rows) {
  if (ranges == nullptr || num_heads < 1 || num_kv_heads < 1 || head_dim < 1 || tp_size < 1 || tp_rank < 0 ||
      tp_rank >= tp_size)
    return MLR_ERR_INVALID;
  const int64_t q_dim = (int64_t)num_heads * head_dim, kv_dim = (int64_t)num_kv_heads * head_dim;
  if (q_dim + 2 * kv_dim > INT32_MAX) return MLR_ERR_INVALID;
  if (num_heads % tp_size != 0) return MLR_ERR_INVALID;  // q heads split evenly
  int64_t kv_rows, kv_id;
  if (tp_size <= num_kv_heads) {
    if (num_kv_heads % tp_size != 0) return MLR_ERR_INVALID;
    kv_rows = kv_dim / tp_size;
    kv_id = tp_rank;
  } else {
    if (tp_size % num_kv_heads != 0) return MLR_ERR_INVALID;
    const int64_t replicas = tp_size / num_kv_heads;
    kv_rows = head_dim;
    kv_id = tp_rank / replicas;
  }
  const int64_t q_rows = q_dim / tp_size;
  const int64_t r[6] = {q_rows * tp_rank,           q_rows * (tp_rank + 1),
                        q_dim + kv_rows * kv_id,    q_dim + kv_rows * (kv_id + 1),
                        q_dim + kv_dim + kv_rows * kv_id, q_dim + kv_dim + kv_rows * (kv_id + 1)};
  for (int i = 0; i < 6; ++i) ranges[i] = (int32_t)r[i];
  if (per_rank_rows) *per_rank_rows = (int32_t)(q_rows + 2 * kv_rows);
  return MLR_OK;
}
