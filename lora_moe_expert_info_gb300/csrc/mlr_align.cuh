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

// Enqueues the align: one launch on the single-block path (below), else the
// four chunked launches.  Workspace holds cnt[G][NB], btotal[NB] (pairs per
// bucket) and bstart[NB+1] (padded bucket starts; bstart[NB] = total); both
// paths leave bstart filled.
int align_launch(const AlignPlan& pl, const int32_t* topk_ids, const int32_t* mapping, int topk,
                 int E, int L, int block_size, int32_t* sorted_ids, int32_t* block_expert,
                 int32_t* block_lora, int32_t* num_post_pad, int64_t capacity, void* workspace,
                 int32_t* d_status, cudaStream_t stream);

// The dense order for the forward on the chunked path, in two parts around the
// caller's scan of the bucket sizes: align_dense_count leaves the per-chunk
// counts (column-scanned) and btotal[NB] (bucket sizes) in the workspace;
// align_dense_scatter then writes each valid pair id to
// dense_sorted[dense_start[b] + its stable rank in bucket b].
int align_dense_count(const AlignPlan& pl, const int32_t* topk_ids, const int32_t* mapping, int topk, int E,
                      int L, void* workspace, int32_t* d_status, cudaStream_t stream);
int align_dense_scatter(const AlignPlan& pl, const int32_t* topk_ids, const int32_t* mapping, int topk, int E,
                        int L, const void* workspace, const uint32_t* dense_start, int32_t* dense_sorted,
                        cudaStream_t stream);


// ---------------------------------------------------------------------------
// Single-block align.  Up to 16384 pairs (16 per thread of a 1024-thread
// block) and 8192 buckets, one block does the whole count / scan / scatter in
// shared memory, which saves the chunked path's launches and its global count
// matrix.  The result is the same canonical stable order.  Its per-pair work
// runs on one SM, so past this size the chunked path is faster (measured on
// the 32768-pair Qwen-like batch: 91 us in one block against 50 us chunked).
constexpr int kAlignBlockThreads = 1024;
constexpr int kAlignBlockMaxItems = 16;
constexpr int64_t kAlignBlockMaxPairs = kAlignBlockThreads * kAlignBlockMaxItems;
constexpr int kAlignBlockMaxBuckets = 8192;
// dynamic shared memory of the one-block kernels, leaving room for their
// static arrays (scan scratch, the plan's rank cache and queue) under 227 KB
constexpr size_t kAlignBlockSmemLimit = 216 * 1024;

// Dynamic shared memory of align_block: cnt[NB+1], start[NB+1] (uint32),
// stage[P], order[P] (uint16).
inline size_t align_block_smem(const AlignPlan& pl) {
  return (size_t)(2 * round_up((int64_t)(pl.NB + 1) * 4, 16) + 2 * round_up(pl.P * 2, 16));
}
// extra: shared memory a caller adds after align_block's (the forward's plan scan)
inline bool align_block_ok(const AlignPlan& pl, size_t extra = 0) {
  return pl.ok && pl.P > 0 && pl.P <= kAlignBlockMaxPairs && pl.NB <= kAlignBlockMaxBuckets &&
         align_block_smem(pl) + extra <= kAlignBlockSmemLimit;
}

// Block-wide exclusive scan of s[0..n) in place; s[n] receives the total.
// Ends with a barrier, so s is ready for every thread on return.
static __device__ void align_block_scan(uint32_t* s, int n) {
  __shared__ uint32_t warp_tot[32];
  const int per = (n + blockDim.x - 1) / blockDim.x;
  const int b0 = min(n, (int)threadIdx.x * per), b1 = min(n, b0 + per);
  uint32_t local = 0;
  for (int b = b0; b < b1; ++b) local += s[b];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t inc = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t v = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += v;
  }
  if (lane == 31) warp_tot[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    const int nw = blockDim.x >> 5;
    uint32_t w = lane < nw ? warp_tot[lane] : 0u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t v = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += v;
    }
    if (lane < nw) warp_tot[lane] = w;
  }
  __syncthreads();
  uint32_t run = inc - local + (warp > 0 ? warp_tot[warp - 1] : 0u);
  for (int b = b0; b < b1; ++b) {
    const uint32_t c = s[b];
    s[b] = run;
    run += c;
  }
  if (threadIdx.x == blockDim.x - 1) s[n] = run;
  __syncthreads();
}

// The whole align in one block of kAlignBlockThreads threads (align_block_ok
// holds).  smem points at align_block_smem bytes of dynamic shared memory.
// On return (after a barrier) cnt holds the exclusive scan of the bucket sizes
// (cnt[NB] = valid pairs).  With dense_out == nullptr, start holds the padded
// bucket starts (start[NB] = total), also copied to bstart_out if given, and the
// outputs are written as by the chunked path.  With dense_out, only the dense
// order is written: dense_out[u] = the u-th pair in bucket order.
struct AlignBlockSmem {
  uint32_t* cnt;    // [NB+1] per-bucket counts, then first slot of each bucket
  uint32_t* start;  // [NB+1] padded bucket starts
  uint16_t* stage;  // [P] pair index by (bucket, round) slot
  uint16_t* order;  // [P] pair index in final (stable) order
};
static __device__ __forceinline__ AlignBlockSmem align_block_carve(unsigned char* smem, int NB, int P) {
  AlignBlockSmem m;
  m.cnt = reinterpret_cast<uint32_t*>(smem);
  m.start = m.cnt + round_up(NB + 1, 4);
  m.stage = reinterpret_cast<uint16_t*>(m.start + round_up(NB + 1, 4));
  m.order = m.stage + round_up(P, 8);
  return m;
}

// Dense order for batches with few buckets (<= kAlignFewBuckets, e.g. one
// expert: a dense projection with per-segment adapters).  Thread t owns the
// contiguous pairs [t * ipt, (t + 1) * ipt); per bucket, a block-wide exclusive
// scan of the per-thread counts gives each thread the place of its first pair
// of that bucket, so pairs land in increasing index inside every bucket
// (stable) without any per-pair search.  On return cnt[b] is the first dense
// row of bucket b and cnt[NB] the number of valid pairs, as after align_block.
constexpr int kAlignFewBuckets = 16;
static __device__ __noinline__ void align_block_few(const int32_t* __restrict__ topk_ids, const int32_t* __restrict__ mapping,
                                       int P, int topk, int E, int L, uint32_t* cnt, int32_t* d_status,
                                       int32_t* __restrict__ dense_out) {
  __shared__ uint32_t wsum[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int C = L + 1, NB = E * C;
  const int ipt = (P + kAlignBlockThreads - 1) / kAlignBlockThreads;  // <= kAlignBlockMaxItems
  const int j0 = tid * ipt;
  uint8_t key[kAlignBlockMaxItems];
  int bad = 0;
#pragma unroll
  for (int i = 0; i < kAlignBlockMaxItems; ++i) {
    key[i] = 0xFF;
    const int j = j0 + i;
    if (i < ipt && j < P) {
      const int e = __ldg(topk_ids + j);
      const int l = __ldg(mapping + j / topk);
      if (e < 0 || e >= E || l < -1 || l >= L) bad |= MLR_STATUS_INDEX;
      else key[i] = (uint8_t)(e * C + l + 1);
    }
  }
  if (bad) set_status(d_status, bad);
  uint32_t off[kAlignFewBuckets];
#pragma unroll
  for (int b = 0; b < kAlignFewBuckets; ++b) {
    off[b] = 0;
    if (b >= NB) continue;  // uniform over the block
    uint32_t mine = 0;
#pragma unroll
    for (int i = 0; i < kAlignBlockMaxItems; ++i) mine += key[i] == b ? 1u : 0u;
    uint32_t inc = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t v = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += v;
    }
    if (lane == 31) wsum[warp] = inc;
    __syncthreads();
    if (warp == 0) {
      uint32_t w = wsum[lane];  // kAlignBlockThreads / 32 == 32 warps
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += v;
      }
      wsum[lane] = w;
      if (lane == 31) cnt[b] = w;  // bucket size
    }
    __syncthreads();
    off[b] = inc - mine + (warp > 0 ? wsum[warp - 1] : 0u);
    __syncthreads();  // wsum is reused by the next bucket
  }
  if (tid == 0) {
    uint32_t run = 0;
    for (int b = 0; b < NB; ++b) {
      const uint32_t n = cnt[b];
      cnt[b] = run;
      run += n;
    }
    cnt[NB] = run;
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < kAlignBlockMaxItems; ++i) {
    const int b = key[i];
    if (b == 0xFF) continue;
    uint32_t o = 0;
#pragma unroll
    for (int q = 0; q < kAlignFewBuckets; ++q)
      if (q == b) o = off[q]++;
    dense_out[cnt[b] + o] = j0 + i;
  }
  __syncthreads();
}

static __device__ void align_block(const int32_t* __restrict__ topk_ids,
                                   const int32_t* __restrict__ mapping, int P, int topk, int E,
                                   int L, int block_size, const AlignBlockSmem& sm,
                                   int32_t* __restrict__ sorted_ids,
                                   int32_t* __restrict__ block_expert, int32_t* __restrict__ block_lora,
                                   int32_t* __restrict__ num_post_pad, uint32_t* __restrict__ bstart_out,
                                   int64_t capacity, int32_t* d_status,
                                   int32_t* __restrict__ dense_out = nullptr) {
  uint32_t* cnt = sm.cnt;
  uint32_t* start = sm.start;
  uint16_t* stage = sm.stage;
  uint16_t* order = sm.order;
  const int tid = threadIdx.x;
  const int C = L + 1, NB = E * C;
  if (dense_out != nullptr && NB <= kAlignFewBuckets) {
    align_block_few(topk_ids, mapping, P, topk, E, L, cnt, d_status, dense_out);
    return;
  }
  for (int b = tid; b <= NB; b += kAlignBlockThreads) cnt[b] = 0u;
  const int rounds = (P + kAlignBlockThreads - 1) / kAlignBlockThreads;
  // Keys of pairs j = it * 1024 + tid; the token j / topk is advanced per round
  // without a division.
  uint32_t ks[kAlignBlockMaxItems];
  int bad = 0;
  {
    const int dq = kAlignBlockThreads / topk, dr = kAlignBlockThreads % topk;
    int tq = tid / topk, tr = tid % topk;
#pragma unroll
    for (int it = 0; it < kAlignBlockMaxItems; ++it) {
      ks[it] = 0xFFFFFFFFu;
      const int j = it * kAlignBlockThreads + tid;
      if (it < rounds && j < P) {
        const int e = __ldg(topk_ids + j);
        const int l = __ldg(mapping + tq);
        if (e < 0 || e >= E || l < -1 || l >= L) bad |= MLR_STATUS_INDEX;
        else ks[it] = (uint32_t)(e * C + l + 1);
      }
      tq += dq;
      tr += dr;
      if (tr >= topk) {
        tr -= topk;
        ++tq;
      }
    }
  }
  if (bad) set_status(d_status, bad);
  __syncthreads();
  // One counting round per 1024 consecutive pairs, separated by barriers, so
  // a bucket's slots follow round order.
#pragma unroll
  for (int it = 0; it < kAlignBlockMaxItems; ++it) {
    if (it < rounds) {
      if (ks[it] != 0xFFFFFFFFu) ks[it] = (ks[it] << 16) | atomicAdd(&cnt[ks[it]], 1u);
      __syncthreads();
    }
  }
  // start[] is kept in units of blocks until the end (no divisions later on)
  for (int b = tid; b < NB; b += kAlignBlockThreads) start[b] = (cnt[b] + block_size - 1) / block_size;
  __syncthreads();
  align_block_scan(cnt, NB);    // cnt[b]: first slot of bucket b in stage / order
  align_block_scan(start, NB);  // start[b]: first block of bucket b
  if (tid == 0 && dense_out == nullptr) {
    const int64_t total = (int64_t)start[NB] * block_size;
    *num_post_pad = (int32_t)total;
    if (total > capacity) set_status(d_status, MLR_STATUS_CAPACITY);
  }
#pragma unroll
  for (int it = 0; it < kAlignBlockMaxItems; ++it)
    if (it < rounds && ks[it] != 0xFFFFFFFFu)
      stage[cnt[ks[it] >> 16] + (ks[it] & 0xFFFFu)] = (uint16_t)(it * kAlignBlockThreads + tid);
  __syncthreads();
  // Final order inside shared memory: the pairs of one round in one bucket are
  // a contiguous run of stage (round = stage value >> 10); each pair's place is
  // the run's start plus the number of run members with a smaller index.
#pragma unroll
  for (int it = 0; it < kAlignBlockMaxItems; ++it) {
    if (it < rounds && ks[it] != 0xFFFFFFFFu) {
      const int k = (int)(ks[it] >> 16);
      const uint32_t j = it * kAlignBlockThreads + tid;
      const int lo = (int)cnt[k], hi = (int)cnt[k + 1];
      const int pos = lo + (int)(ks[it] & 0xFFFFu);
      int less = 0, m = pos - 1;
      while (m >= lo && (stage[m] >> 10) == (uint32_t)it) {
        less += stage[m] < j;
        --m;
      }
      const int run_start = m + 1;
      for (m = pos + 1; m < hi && (stage[m] >> 10) == (uint32_t)it; ++m) less += stage[m] < j;
      order[run_start + less] = (uint16_t)j;
    }
  }
  __syncthreads();
  if (dense_out != nullptr) {
    // the dense order (no padding, no labels): order itself, written out
    for (int u = tid; u < (int)cnt[NB]; u += kAlignBlockThreads) dense_out[u] = order[u];
    __syncthreads();
    return;
  }
  // Output.  Labels, and an owner table block -> bucket in stage (no longer
  // needed; a bucket has at least as many pairs as blocks, so P entries hold
  // every block), are written bucket-parallel; sorted ids and pad sentinels
  // are then written position-parallel, coalesced.  Positions are below
  // P + NB * block_size < 2^31.
  const int64_t cap64 = capacity < INT32_MAX ? capacity : INT32_MAX;
  const int cap = (int)cap64, cap_blocks = (int)(cap64 / block_size);
  for (int b = tid; b < NB; b += kAlignBlockThreads) {
    const int kb0 = (int)start[b], kb1 = (int)start[b + 1];
    if (kb1 == kb0) continue;
    const int expert = b / C, lora = b - expert * C - 1;
    for (int blk = kb0; blk < kb1; ++blk) {
      stage[blk] = (uint16_t)b;
      if (blk < cap_blocks) {
        block_expert[blk] = expert;
        block_lora[blk] = lora;
      }
    }
  }
  __syncthreads();
  {
    const int total = min((int)start[NB] * block_size, cap);
    // position q = blk * block_size + rem, advanced by 1024 without a division
    const int dq = kAlignBlockThreads / block_size, dr = kAlignBlockThreads % block_size;
    int blk = tid / block_size, rem = tid % block_size;
    for (int q = tid; q < total; q += kAlignBlockThreads) {
      const int b = stage[blk];
      const int i = (blk - (int)start[b]) * block_size + rem;
      const int lo = (int)cnt[b];
      sorted_ids[q] = i < (int)cnt[b + 1] - lo ? (int32_t)order[lo + i] : P;
      blk += dq;
      rem += dr;
      if (rem >= block_size) {
        rem -= block_size;
        ++blk;
      }
    }
  }
  __syncthreads();
  for (int b = tid; b <= NB; b += kAlignBlockThreads) {
    start[b] *= (uint32_t)block_size;  // padded start of bucket b, in pairs
    if (bstart_out != nullptr) bstart_out[b] = start[b];
  }
  __syncthreads();
}

}  // namespace mlr
