// ep.cu -- expert-parallel dispatch and combine of the LoRA MoE layer.
//
// The experts are split over n ranks in equal contiguous ranges (rank d owns
// experts [d*E/n, (d+1)*E/n)).  The pages name expert parallelism only as the
// multi-GPU form other PRs build on (the DeepEP dispatch among the quant-info
// page's related PRs; the TP/EP question in the LoRA-MoE page's review); the
// steps here are the plain ones:
//   dispatch  every pair p = t*K + k with expert e in [0, E) goes to rank
//             e / (E/n); each rank's pairs are packed in increasing p into the
//             send buffers (x row, expert id relative to the rank's first
//             expert, routing weight, adapter), and pair_pos[p] records where
//   (exchange and the owner's forward are the caller's: an all-to-all of the
//    packed rows, then fused_moe_lora_forward with top-1 over the local
//    experts, then the reverse all-to-all of the weighted output rows)
//   combine   y_t = sum over k, in increasing k, of the returned rows of t's
//             pairs, in fp32 (bit-identical between runs)
//
// Launches of the dispatch: a count over blocks of 1024 pairs (per warp and
// destination, stable ranks from __match_any_sync), a one-block scan into the
// per-block send offsets, and a scatter that recomputes the same ranks and
// writes the send order and pair_pos; a pack kernel then copies the x rows
// (one warp per row, 16-byte lanes) and the per-row metadata.
#include "mlr_profile.cuh"

namespace mlr {
namespace {

constexpr int kEpThreads = 1024;  // pairs per block of the count / scatter
constexpr int kEpWarps = kEpThreads / 32;
constexpr int kEpMaxRanks = 64;
constexpr int kPackThreads = 256;

// Destination rank of pair p, or -1 for an expert id outside [0, E).
__device__ __forceinline__ int ep_dest(const int32_t* __restrict__ ids, int64_t p, int64_t P, int E, int per) {
  if (p >= P) return -2;  // past the end: no pair
  const int e = __ldg(ids + p);
  return (e < 0 || e >= E) ? -1 : e / per;
}

// Per warp: the stable rank of this lane's pair among the warp's lanes with
// the same destination, and (lane d) the warp's count for destination d.
__device__ __forceinline__ void ep_warp_ranks(int dest, int lane, int n_ranks, int* rank_in_warp,
                                              int* warp_count_of_lane) {
  const unsigned same = __match_any_sync(0xffffffffu, dest);
  *rank_in_warp = __popc(same & ((1u << lane) - 1u));
  // warp_count_of_lane: count of destination `lane` (and lane + 32) in this warp
  int c0 = 0, c1 = 0;
  for (int d = 0; d < n_ranks; ++d) {
    const int c = __popc(__ballot_sync(0xffffffffu, dest == d));
    if (d == lane) c0 = c;
    if (d == lane + 32) c1 = c;
  }
  warp_count_of_lane[0] = c0;
  warp_count_of_lane[1] = c1;
}

__global__ void __launch_bounds__(kEpThreads)
ep_count_kernel(const int32_t* __restrict__ ids, int64_t P, int E, int per, int n_ranks,
                int32_t* __restrict__ cnt /* [G][n_ranks] */, int32_t* d_status) {
  __shared__ int wc[kEpWarps][kEpMaxRanks];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t p = (int64_t)blockIdx.x * kEpThreads + threadIdx.x;
  const int dest = ep_dest(ids, p, P, E, per);
  if (dest == -1) set_status(d_status, MLR_STATUS_INDEX);
  int r, c[2];
  ep_warp_ranks(dest, lane, n_ranks, &r, c);
  wc[warp][lane] = c[0];
  if (kEpMaxRanks > 32) wc[warp][lane + 32] = c[1];
  __syncthreads();
  for (int d = threadIdx.x; d < n_ranks; d += kEpThreads) {
    int s = 0;
    for (int w = 0; w < kEpWarps; ++w) s += wc[w][d];
    cnt[(int64_t)blockIdx.x * n_ranks + d] = s;
  }
}

// One block: off[g][d] = start of destination d + pairs of d in blocks < g;
// send_counts[d]; total[0] = all valid pairs.
__global__ void __launch_bounds__(kEpThreads)
ep_scan_kernel(int32_t* __restrict__ cnt /* in: counts, out: offsets */, int G, int n_ranks,
               int32_t* __restrict__ send_counts, int32_t* __restrict__ total) {
  __shared__ int dtot[kEpMaxRanks];
  __shared__ int part[kEpThreads];
  // per destination: a block-wide scan over the G block counts
  for (int d = 0; d < n_ranks; ++d) {
    const int per_t = (G + kEpThreads - 1) / kEpThreads;
    const int g0 = min(G, (int)threadIdx.x * per_t), g1 = min(G, g0 + per_t);
    int local = 0;
    for (int g = g0; g < g1; ++g) local += cnt[(int64_t)g * n_ranks + d];
    part[threadIdx.x] = local;
    __syncthreads();
    // Hillis-Steele inclusive scan of part (kEpThreads entries)
    for (int o = 1; o < kEpThreads; o <<= 1) {
      const int v = threadIdx.x >= o ? part[threadIdx.x - o] : 0;
      __syncthreads();
      part[threadIdx.x] += v;
      __syncthreads();
    }
    int run = part[threadIdx.x] - local;
    for (int g = g0; g < g1; ++g) {
      const int v = cnt[(int64_t)g * n_ranks + d];
      cnt[(int64_t)g * n_ranks + d] = run;
      run += v;
    }
    if (threadIdx.x == kEpThreads - 1) dtot[d] = part[kEpThreads - 1];
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    int run = 0;
    for (int d = 0; d < n_ranks; ++d) {
      send_counts[d] = dtot[d];
      const int v = dtot[d];
      dtot[d] = run;
      run += v;
    }
    total[0] = run;
  }
  __syncthreads();
  for (int64_t i = threadIdx.x; i < (int64_t)G * n_ranks; i += kEpThreads) cnt[i] += dtot[i % n_ranks];
}

__global__ void __launch_bounds__(kEpThreads)
ep_scatter_kernel(const int32_t* __restrict__ ids, int64_t P, int E, int per, int n_ranks,
                  const int32_t* __restrict__ off /* [G][n_ranks] */, int32_t* __restrict__ send_pair,
                  int32_t* __restrict__ pair_pos) {
  __shared__ int wc[kEpWarps][kEpMaxRanks];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t p = (int64_t)blockIdx.x * kEpThreads + threadIdx.x;
  const int dest = ep_dest(ids, p, P, E, per);
  int r, c[2];
  ep_warp_ranks(dest, lane, n_ranks, &r, c);
  wc[warp][lane] = c[0];
  if (kEpMaxRanks > 32) wc[warp][lane + 32] = c[1];
  __syncthreads();
  if (dest >= 0) {
    int before = 0;  // pairs of this destination in earlier warps of the block
    for (int w = 0; w < warp; ++w) before += wc[w][dest];
    const int q = off[(int64_t)blockIdx.x * n_ranks + dest] + before + r;
    send_pair[q] = (int32_t)p;
    pair_pos[p] = q;
  } else if (dest == -1) {
    pair_pos[p] = -1;
  }
}

// One warp per send row: the x row of the pair's token, its expert relative to
// the destination's first expert, its weight and its token's adapter.
__global__ void __launch_bounds__(kPackThreads)
ep_pack_kernel(const uint16_t* __restrict__ x, const int32_t* __restrict__ ids, const float* __restrict__ w,
               const int32_t* __restrict__ mapping, const int32_t* __restrict__ send_pair,
               const int32_t* __restrict__ total, int K, int H, int per, uint16_t* __restrict__ send_x,
               int32_t* __restrict__ send_expert, float* __restrict__ send_weight, int32_t* __restrict__ send_lora) {
  const int64_t n = *total;
  const int lane = threadIdx.x & 31;
  const int64_t wpb = kPackThreads / 32;
  for (int64_t i = (int64_t)blockIdx.x * wpb + (threadIdx.x >> 5); i < n; i += (int64_t)gridDim.x * wpb) {
    const int64_t p = send_pair[i];
    const int64_t t = p / K;
    const uint4* src = reinterpret_cast<const uint4*>(x + t * H);
    uint4* dst = reinterpret_cast<uint4*>(send_x + i * H);
    for (int c = lane; c < H / 8; c += 32) dst[c] = __ldg(src + c);
    if (lane == 0) {
      const int e = ids[p];
      send_expert[i] = e % per;
      send_weight[i] = w[p];
      send_lora[i] = mapping[t];
    }
  }
}

// y[t] = sum over k (increasing) of rows[pair_pos[t*K + k]], skipping -1; fp32
// sums of bf16 rows, one thread per 8 consecutive columns of a token.
__global__ void ep_combine_kernel(const uint16_t* __restrict__ rows, const int32_t* __restrict__ pair_pos,
                                  int64_t T, int K, int H, uint16_t* __restrict__ y) {
  const int g8 = H / 8;
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= T * g8) return;
  const int64_t t = i / g8;
  const int c = (int)(i - t * g8) * 8;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  // up to 8 pairs' rows in flight before any is added; the sum runs in increasing k
  for (int k0 = 0; k0 < K; k0 += 8) {
    uint4 v[8];
    int q[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      q[j] = k0 + j < K ? __ldg(pair_pos + t * K + k0 + j) : -1;
      v[j] = q[j] >= 0 ? __ldg(reinterpret_cast<const uint4*>(rows + (int64_t)q[j] * H + c)) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (q[j] < 0) continue;
      const uint32_t wv[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        acc[2 * u] += __uint_as_float(wv[u] << 16);
        acc[2 * u + 1] += __uint_as_float(wv[u] & 0xffff0000u);
      }
    }
  }
  uint4 o;
  o.x = (uint32_t)f32_to_bf16_bits(acc[0]) | ((uint32_t)f32_to_bf16_bits(acc[1]) << 16);
  o.y = (uint32_t)f32_to_bf16_bits(acc[2]) | ((uint32_t)f32_to_bf16_bits(acc[3]) << 16);
  o.z = (uint32_t)f32_to_bf16_bits(acc[4]) | ((uint32_t)f32_to_bf16_bits(acc[5]) << 16);
  o.w = (uint32_t)f32_to_bf16_bits(acc[6]) | ((uint32_t)f32_to_bf16_bits(acc[7]) << 16);
  *reinterpret_cast<uint4*>(y + t * H + c) = o;
}

struct EpLayout {
  bool ok;
  int64_t P, G;
  int64_t o_cnt, o_pair, o_total, total;
};

EpLayout ep_layout(int32_t T, int32_t K, int32_t n_ranks) {
  EpLayout f{};
  f.ok = false;
  if (T < 0 || K < 1 || n_ranks < 1 || n_ranks > kEpMaxRanks) return f;
  f.P = (int64_t)T * K;
  if (f.P >= INT32_MAX) return f;
  f.G = ceil_div(f.P, kEpThreads);
  int64_t o = 0;
  auto take = [&](int64_t bytes) { const int64_t r = o; o += round_up(bytes > 0 ? bytes : 1, 256); return r; };
  f.o_cnt = take(f.G * n_ranks * 4);
  f.o_pair = take(f.P * 4);
  f.o_total = take(16);
  f.total = o;
  f.ok = true;
  return f;
}

}  // namespace
}  // namespace mlr

extern "C" size_t moe_lora_ep_workspace_bytes(int32_t num_tokens, int32_t topk, int32_t n_ranks) {
  const mlr::EpLayout f = mlr::ep_layout(num_tokens, topk, n_ranks);
  return f.ok ? (size_t)f.total : 0;
}

extern "C" int moe_lora_ep_dispatch(const mlr_bf16* x, const int32_t* topk_ids, const float* topk_weights,
                                    const int32_t* token_lora_mapping, int32_t num_tokens, int32_t topk,
                                    int32_t hidden, int32_t num_experts, int32_t n_ranks, mlr_bf16* send_x,
                                    int32_t* send_expert, float* send_weight, int32_t* send_lora,
                                    int32_t* send_counts, int32_t* pair_pos, void* workspace, size_t ws_bytes,
                                    int32_t* d_status, void* stream_) {
  using namespace mlr;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  const EpLayout f = ep_layout(num_tokens, topk, n_ranks);
  if (!f.ok || hidden < 8 || hidden % 8 != 0 || num_experts < 1) {
    if (n_ranks > kEpMaxRanks && num_tokens >= 0 && topk >= 1) return MLR_ERR_UNSUPPORTED;
    return MLR_ERR_INVALID;
  }
  if (num_experts % n_ranks != 0) return MLR_ERR_INVALID;
  if (send_counts == nullptr) return MLR_ERR_INVALID;
  if (f.P > 0) {
    const void* need[] = {x, topk_ids, topk_weights, token_lora_mapping, send_x, send_expert, send_weight,
                          send_lora, pair_pos};
    for (const void* q : need)
      if (q == nullptr) return MLR_ERR_INVALID;
    if ((reinterpret_cast<uintptr_t>(x) & 15) != 0 || (reinterpret_cast<uintptr_t>(send_x) & 15) != 0)
      return MLR_ERR_INVALID;
  }
  if (workspace == nullptr || ws_bytes < (size_t)f.total) return MLR_ERR_CAPACITY;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255) != 0) return MLR_ERR_INVALID;
  char* ws = static_cast<char*>(workspace);
  int32_t* cnt = reinterpret_cast<int32_t*>(ws + f.o_cnt);
  int32_t* send_pair = reinterpret_cast<int32_t*>(ws + f.o_pair);
  int32_t* total = reinterpret_cast<int32_t*>(ws + f.o_total);
  const int per = num_experts / n_ranks;
  if (f.G > 0) {
    ep_count_kernel<<<(unsigned)f.G, kEpThreads, 0, stream>>>(topk_ids, f.P, num_experts, per, n_ranks, cnt,
                                                               d_status);
    MLR_CHECK_LAUNCH();
    note_launch();
  }
  ep_scan_kernel<<<1, kEpThreads, 0, stream>>>(cnt, (int)f.G, n_ranks, send_counts, total);
  MLR_CHECK_LAUNCH();
  note_launch();
  if (f.G > 0) {
    ep_scatter_kernel<<<(unsigned)f.G, kEpThreads, 0, stream>>>(topk_ids, f.P, num_experts, per, n_ranks, cnt,
                                                                 send_pair, pair_pos);
    MLR_CHECK_LAUNCH();
    note_launch();
    const int64_t blocks = ceil_div(f.P, kPackThreads / 32);
    const unsigned grid = (unsigned)(blocks < 8 * 152 ? blocks : 8 * 152);
    ep_pack_kernel<<<grid, kPackThreads, 0, stream>>>(
        reinterpret_cast<const uint16_t*>(x), topk_ids, topk_weights, token_lora_mapping, send_pair, total, topk,
        hidden, per, reinterpret_cast<uint16_t*>(send_x), send_expert, send_weight, send_lora);
    MLR_CHECK_LAUNCH();
    note_launch();
  }
  return MLR_OK;
}

extern "C" int moe_lora_ep_combine(const mlr_bf16* rows, const int32_t* pair_pos, int32_t num_tokens, int32_t topk,
                                   int32_t hidden, mlr_bf16* y, void* stream_) {
  using namespace mlr;
  if (num_tokens < 0 || topk < 1 || hidden < 8 || hidden % 8 != 0) return MLR_ERR_INVALID;
  const int64_t n8 = (int64_t)num_tokens * (hidden / 8);
  if (n8 == 0) return MLR_OK;
  if (pair_pos == nullptr || y == nullptr) return MLR_ERR_INVALID;
  if ((reinterpret_cast<uintptr_t>(y) & 15) != 0 || (rows != nullptr && (reinterpret_cast<uintptr_t>(rows) & 15) != 0))
    return MLR_ERR_INVALID;
  ep_combine_kernel<<<(unsigned)ceil_div(n8, 256), 256, 0, static_cast<cudaStream_t>(stream_)>>>(
      reinterpret_cast<const uint16_t*>(rows), pair_pos, num_tokens, topk, hidden, reinterpret_cast<uint16_t*>(y));
  MLR_CHECK_LAUNCH();
  note_launch();
  return MLR_OK;
}
