// batch_info.cu -- moe_lora_batch_info: once per batch, expand request segments
// into token_lora_mapping and adapter_enabled (sglang PR #24160 page, 实现拆解
// items 1-3 and the MoELoRABatchInfo dataclass in 关键源码片段).
//
// One launch.  Blocks 0..nt-1 each own a tile of 1024 consecutive tokens: the
// block finds the first and last request segment of its tile with a
// block-cooperative 256-way search, stages that run of seg_indptr /
// weight_indices in shared memory and
// every thread resolves 4 consecutive tokens there (one 16-byte store).  The
// last block validates seg_indptr, the max_len hint and the adapter ids, and
// writes all num_loras entries of adapter_enabled from a shared bit set.
#include "mlr_profile.cuh"

namespace mlr {
namespace {

constexpr int kThreads = 256;
constexpr int kTokPerThread = 4;
constexpr int kTile = kThreads * kTokPerThread;
constexpr int kStaged = 2048;               // segments staged per tile
constexpr int kMaxLoras = 65536;            // adapter_enabled bit set: 8 KB

// Block-wide search for the segments of two tokens ta <= tb: the largest i in
// [0, bs - 1] with indptr[i] <= t, for t = ta and t = tb (indptr assumed
// non-decreasing; any result stays in [0, bs - 1] otherwise).  Each round the
// block samples kThreads evenly spaced entries of the remaining range and
// counts those <= t, which narrows the range kThreads-fold: two or three
// rounds of one load per thread instead of a serial binary search of
// log2(bs) dependent loads.  All threads of the block call it.
__device__ __forceinline__ void block_seg_search2(const int32_t* __restrict__ indptr, int bs, int ta, int tb,
                                                  int* ra, int* rb) {
  int a0 = 0, b0 = bs - 1, a1 = 0, b1 = bs - 1;  // inclusive ranges of the two answers
  while (true) {
    const int na = b0 - a0 + 1, nb = b1 - a1 + 1;
    if (na <= 1 && nb <= 1) break;
    const int sa = (na + kThreads - 1) / kThreads, sb = (nb + kThreads - 1) / kThreads;  // strides
    const int ca = a0 + (int)threadIdx.x * sa, cb = a1 + (int)threadIdx.x * sb;
    const bool pa = na > 1 && ca <= b0 && __ldg(indptr + ca) <= ta;
    const bool pb = nb > 1 && cb <= b1 && __ldg(indptr + cb) <= tb;
    const int ka = __syncthreads_count(pa), kb = __syncthreads_count(pb);
    if (na > 1) {
      const int lo = a0 + (max(ka, 1) - 1) * sa;  // the answer lies in [lo, lo + sa - 1]
      a0 = lo;
      b0 = min(b0, lo + sa - 1);
    }
    if (nb > 1) {
      const int lo = a1 + (max(kb, 1) - 1) * sb;
      a1 = lo;
      b1 = min(b1, lo + sb - 1);
    }
  }
  *ra = a0;
  *rb = a1;
}

// largest i in [lo, hi] with indptr[i] <= t  (indptr assumed non-decreasing)
__device__ __forceinline__ int seg_search(const int32_t* __restrict__ indptr, int lo, int hi, int t) {
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(indptr + mid) <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__global__ void __launch_bounds__(kThreads)
batch_info_kernel(const int32_t* __restrict__ seg_indptr, const int32_t* __restrict__ weight_indices,
                  const int32_t* __restrict__ lora_ranks, int bs, int num_loras, int num_tokens,
                  int max_len, int32_t* __restrict__ mapping, int32_t* __restrict__ enabled,
                  int32_t* d_status, int vec_ok) {
  pdl_wait();  // the predecessor on the stream has completed
  pdl_trigger();
  __shared__ int32_t s_ptr[kStaged + 1];
  __shared__ int32_t s_wi[kStaged];
  __shared__ uint32_t s_bits[kMaxLoras / 32];
  __shared__ int s_bad;

  const int ntile = (int)ceil_div(num_tokens, kTile);
  if ((int)blockIdx.x == ntile) {
    // ---- validation and adapter_enabled ----
    const int nwords = (num_loras + 31) >> 5;
    for (int w = threadIdx.x; w < nwords; w += blockDim.x) s_bits[w] = 0u;
    if (threadIdx.x == 0) s_bad = 0;
    __syncthreads();
    int bad = 0;
    // kVBatch segments per thread per round, their loads issued together
    constexpr int kVBatch = 8;
    for (int i0 = 0; i0 < bs; i0 += kVBatch * kThreads) {
      int a[kVBatch], b[kVBatch], l[kVBatch];
#pragma unroll
      for (int q = 0; q < kVBatch; ++q) {
        const int i = i0 + q * kThreads + (int)threadIdx.x;
        const int ic = i < bs ? i : 0;
        a[q] = __ldg(seg_indptr + ic);
        b[q] = __ldg(seg_indptr + ic + 1);
        l[q] = __ldg(weight_indices + ic);
      }
#pragma unroll
      for (int q = 0; q < kVBatch; ++q) {
        if (i0 + q * kThreads + (int)threadIdx.x >= bs) continue;
        if (b[q] < a[q]) bad |= MLR_STATUS_BAD_INDPTR;
        if (max_len > 0 && b[q] - a[q] > max_len) bad |= MLR_STATUS_UNDERCOVERED;
        if (l[q] < -1 || l[q] >= num_loras) bad |= MLR_STATUS_INDEX;
        else if (l[q] >= 0) atomicOr(&s_bits[l[q] >> 5], 1u << (l[q] & 31));
      }
    }
    if (threadIdx.x == 0 && (seg_indptr[0] != 0 || seg_indptr[bs] != num_tokens))
      bad |= MLR_STATUS_BAD_INDPTR;
    if (bad) atomicOr(&s_bad, bad);
    __syncthreads();
    for (int l = threadIdx.x; l < num_loras; l += blockDim.x) {
      const bool used = (s_bits[l >> 5] >> (l & 31)) & 1u;
      enabled[l] = (used && lora_ranks[l] > 0) ? 1 : 0;
    }
    if (threadIdx.x == 0) set_status(d_status, s_bad);
    return;
  }

  // ---- token tile ----
  const int t0 = blockIdx.x * kTile;
  const int t_last = min(num_tokens, t0 + kTile) - 1;
  int lo, hi;
  block_seg_search2(seg_indptr, bs, t0, t_last, &lo, &hi);
  const int n = hi - lo + 1;
  const bool staged = (n >= 1 && n <= kStaged);
  if (staged) {
    for (int j = threadIdx.x; j <= n; j += blockDim.x) s_ptr[j] = seg_indptr[lo + j];
    for (int j = threadIdx.x; j < n; j += blockDim.x) s_wi[j] = weight_indices[lo + j];
  }
  __syncthreads();

  const int t = t0 + threadIdx.x * kTokPerThread;
  if (t >= num_tokens) return;
  int v[kTokPerThread];
  if (staged) {
    int j = 0, jh = n - 1;
    while (j < jh) {  // largest j with s_ptr[j] <= t
      const int mid = (j + jh + 1) >> 1;
      if (s_ptr[mid] <= t) j = mid; else jh = mid - 1;
    }
#pragma unroll
    for (int q = 0; q < kTokPerThread; ++q) {
      while (j + 1 < n && s_ptr[j + 1] <= t + q) ++j;
      v[q] = s_wi[j];
    }
  } else {
#pragma unroll
    for (int q = 0; q < kTokPerThread; ++q)
      v[q] = (t + q < num_tokens) ? __ldg(weight_indices + seg_search(seg_indptr, 0, bs - 1, t + q)) : 0;
  }
  if (vec_ok && t + kTokPerThread <= num_tokens) {
    *reinterpret_cast<int4*>(mapping + t) = make_int4(v[0], v[1], v[2], v[3]);
  } else {
#pragma unroll
    for (int q = 0; q < kTokPerThread; ++q)
      if (t + q < num_tokens) mapping[t + q] = v[q];
  }
}

}  // namespace
}  // namespace mlr

extern "C" int moe_lora_batch_info(const int32_t* seg_indptr, const int32_t* weight_indices,
                                   const int32_t* lora_ranks, int32_t bs, int32_t num_loras,
                                   int32_t num_tokens, int32_t max_len,
                                   int32_t* token_lora_mapping, int32_t* adapter_enabled,
                                   int32_t* d_status, void* stream) {
  using namespace mlr;
  if (bs < 0 || num_loras < 0 || num_tokens < 0 || max_len < 0) return MLR_ERR_INVALID;
  if (num_loras > kMaxLoras) return MLR_ERR_UNSUPPORTED;
  if (seg_indptr == nullptr) return MLR_ERR_INVALID;
  if (bs > 0 && weight_indices == nullptr) return MLR_ERR_INVALID;
  if (num_loras > 0 && (lora_ranks == nullptr || adapter_enabled == nullptr)) return MLR_ERR_INVALID;
  if (num_tokens > 0 && (token_lora_mapping == nullptr || bs == 0)) return MLR_ERR_INVALID;
  if (max_len > 0 && (int64_t)bs * (int64_t)max_len < (int64_t)num_tokens) return MLR_ERR_UNDERCOVERED;
  const int ntile = (int)ceil_div(num_tokens, kTile);
  const int vec_ok = (reinterpret_cast<uintptr_t>(token_lora_mapping) % 16) == 0;
  if (launch_pdl(batch_info_kernel, dim3(ntile + 1), dim3(kThreads), 0, static_cast<cudaStream_t>(stream), 
      seg_indptr, weight_indices, lora_ranks, bs, num_loras, num_tokens, max_len,
      token_lora_mapping, adapter_enabled, d_status, vec_ok) != cudaSuccess) return MLR_ERR_CUDA;
  MLR_CHECK_LAUNCH();
  note_launch();
  return MLR_OK;
}
