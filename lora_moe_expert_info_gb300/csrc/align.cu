// align.cu -- moe_lora_align: bucket (token, slot) pairs by (expert, adapter),
// stable, each bucket padded to block_size (sglang PR #14105 page, 实现拆解:
// moe_lora_align_block_size "sorts tokens by LoRA adapter and expert id").
//
// key(p) = e * (L+1) + (lora + 1); NB = E * (L+1) buckets.  Up to
// kAlignBlockMaxPairs (16384) pairs and kAlignBlockMaxBuckets (8192) buckets,
// one block does everything in shared memory (align_block).
// Otherwise pairs are split into G contiguous chunks of up to 32768 pairs and
// four launches follow:
//   1. count    : per chunk, a shared-memory histogram over NB buckets
//                 -> cnt[g][b]
//   2. colscan  : per bucket, exclusive prefix over chunks (in place) and the
//                 bucket total (32 buckets x 32 chunk segments per block)
//   3. bktscan  : one block, exclusive scan of the padded totals in shared
//                 memory -> bucket starts and num_tokens_post_pad
//   4. scatter  : per chunk, stable local ranks and the final placement
//                 (plus the pad sentinels and the per-block expert/adapter ids)
// When two bucket arrays and a chunk fit in shared memory (NB up to about
// 20000), the scatter scans the padded totals itself (launch 3 is skipped)
// and keeps every bucket's global base in shared memory.
// Stability inside a chunk: pairs are visited in rounds of 1024 consecutive
// indices separated by barriers, so a bucket's slots follow round order; the
// few same-round neighbours of a pair are re-ranked by index when it is placed.
#include "mlr_align.cuh"
#include "mlr_profile.cuh"

namespace mlr {
namespace {

constexpr int kThreads = 1024;
constexpr int kMaxItems = 32;                         // pairs per thread per chunk
constexpr int kMaxChunk = kThreads * kMaxItems;       // 32768 (fits uint16 indices)
constexpr int kLoadBatch = 8;                         // pairs whose loads a thread issues together
constexpr size_t kSmemLimit = 227 * 1024;             // dynamic shared memory per block

// The current device, or -1 (per-device caches of the launch set-up).
int current_device_id() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -1;
  return dev;
}

// SMs of the current device (148 when it cannot be read, e.g. without a GPU).
int device_sm_count() {
  static int n[64] = {};
  const int dev = current_device_id();
  if (dev < 0) return 148;
  if (n[dev] == 0) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = 148;
    n[dev] = v;
  }
  return n[dev];
}

// Token of this thread's pair j = it * kThreads + tid of a chunk, advanced one
// round (kThreads pairs) at a time without a division: t = tq, tr = its slot.
struct TokenCursor {
  int tq, tr, dq, dr, topk;
  __device__ __forceinline__ TokenCursor(int64_t p0, int topk_) : topk(topk_) {
    const int64_t p = p0 + threadIdx.x;  // < 2^31: align_plan bounds P
    tq = (int)(p / topk);
    tr = (int)(p - (int64_t)tq * topk);
    dq = kThreads / topk;
    dr = kThreads % topk;
  }
  __device__ __forceinline__ void next() {
    tq += dq;
    tr += dr;
    if (tr >= topk) {
      tr -= topk;
      ++tq;
    }
  }
};

// Keys of this thread's pairs j = (bt + i) * kThreads + tid, i < kLoadBatch, of
// the chunk starting at pair p0 with n pairs (-1 past the end or for an id out
// of range, which also flags `bad`).  All loads are issued before any is used;
// cur holds the token of pair (bt * kThreads + tid) and is advanced past the batch.
__device__ __forceinline__ void align_load_keys(const int32_t* __restrict__ topk_ids,
                                                const int32_t* __restrict__ mapping, int64_t p0, int n, int bt,
                                                TokenCursor& cur, int E, int C, int L, int (&key)[kLoadBatch],
                                                int& bad) {
  int ev[kLoadBatch], lv[kLoadBatch];
#pragma unroll
  for (int i = 0; i < kLoadBatch; ++i) {
    const int j = (bt + i) * kThreads + (int)threadIdx.x;
    const bool in = j < n;
    ev[i] = __ldg(topk_ids + p0 + (in ? j : 0));
    lv[i] = __ldg(mapping + (in ? cur.tq : 0));
    cur.next();
  }
#pragma unroll
  for (int i = 0; i < kLoadBatch; ++i) {
    const int j = (bt + i) * kThreads + (int)threadIdx.x;
    key[i] = -1;
    if (j < n) {
      if (ev[i] < 0 || ev[i] >= E || lv[i] < -1 || lv[i] >= L) bad |= MLR_STATUS_INDEX;
      else key[i] = ev[i] * C + lv[i] + 1;
    }
  }
}
constexpr int kColWarps = 32;  // chunk segments per bucket in the column scan
constexpr int kColThreads = 32 * kColWarps;

__global__ void __launch_bounds__(kThreads, 2)  // two blocks per SM: 32 registers
align_count_kernel(const int32_t* __restrict__ topk_ids, const int32_t* __restrict__ mapping,
                   int64_t P, int topk, int E, int L, int chunk, uint32_t* __restrict__ cnt,
                   int32_t* d_status) {
  pdl_wait();  // the predecessor on the stream has completed
  pdl_trigger();
  extern __shared__ uint32_t hist[];
  const int C = L + 1, NB = E * C;
  for (int b = threadIdx.x; b < NB; b += blockDim.x) hist[b] = 0u;
  __syncthreads();
  const int64_t p0 = (int64_t)blockIdx.x * chunk;
  const int n = (int)(P - p0 < chunk ? P - p0 : chunk);
  int bad = 0;
  // keys in batches of kLoadBatch pairs: the batch's loads are issued together
  // (unconditionally, past-the-end lanes reading pair p0), then counted
  TokenCursor cur(p0, topk);
#pragma unroll
  for (int bt = 0; bt < kMaxItems; bt += kLoadBatch) {
    int key[kLoadBatch];
    align_load_keys(topk_ids, mapping, p0, n, bt, cur, E, C, L, key, bad);
#pragma unroll
    for (int i = 0; i < kLoadBatch; ++i)
      if (key[i] >= 0) atomicAdd(&hist[key[i]], 1u);
  }
  if (bad) set_status(d_status, bad);
  __syncthreads();
  uint32_t* row = cnt + (int64_t)blockIdx.x * NB;
  for (int b = threadIdx.x; b < NB; b += blockDim.x) row[b] = hist[b];
}

// Per bucket, the exclusive prefix of its counts over the chunks, in place,
// and its total.  A block takes 32 buckets (one per lane) and splits the G
// chunks over its 32 warps: each thread sums its segment (loads in flight
// together), the 32 segment sums of a bucket are scanned in shared memory,
// then each thread rewrites its segment.
__global__ void __launch_bounds__(kColThreads)
align_colscan_kernel(uint32_t* __restrict__ cnt, int G, int NB, uint32_t* __restrict__ btotal) {
  pdl_wait();  // the predecessor on the stream has completed
  pdl_trigger();
  __shared__ uint32_t part[kColWarps][33];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int b = blockIdx.x * 32 + lane;
  const int seg = (G + kColWarps - 1) / kColWarps;
  const int g0 = min(G, w * seg), g1 = min(G, g0 + seg);
  uint32_t local = 0;
  if (b < NB) {
#pragma unroll 8
    for (int g = g0; g < g1; ++g) local += cnt[(int64_t)g * NB + b];
  }
  part[w][lane] = local;
  __syncthreads();
  if (w == 0) {
    uint32_t run = 0;
    for (int q = 0; q < kColWarps; ++q) {
      const uint32_t v = part[q][lane];
      part[q][lane] = run;
      run += v;
    }
    if (b < NB) btotal[b] = run;
  }
  __syncthreads();
  uint32_t run = part[w][lane];
  if (b < NB) {
    for (int g = g0; g < g1; ++g) {
      const uint32_t c = cnt[(int64_t)g * NB + b];
      cnt[(int64_t)g * NB + b] = run;
      run += c;
    }
  }
}

// One block: the padded bucket totals are loaded (coalesced) into shared
// memory, scanned there, and written out as the padded bucket starts.
// Dynamic shared memory: (NB + 1) uint32.
__global__ void __launch_bounds__(kThreads)
align_bucketscan_kernel(const uint32_t* __restrict__ btotal, int NB, int block_size,
                        uint32_t* __restrict__ bstart, int32_t* __restrict__ num_post_pad,
                        int64_t capacity, int32_t* d_status) {
  pdl_wait();  // the predecessor on the stream has completed
  pdl_trigger();
  extern __shared__ uint32_t sb[];
  for (int b = threadIdx.x; b < NB; b += blockDim.x)
    sb[b] = (btotal[b] + block_size - 1) / block_size * block_size;
  __syncthreads();
  align_block_scan(sb, NB);  // sb[NB] = total
  for (int b = threadIdx.x; b <= NB; b += blockDim.x) bstart[b] = sb[b];
  if (threadIdx.x == 0) {
    const uint32_t run = sb[NB];
    *num_post_pad = (int32_t)run;
    if ((int64_t)run > capacity) set_status(d_status, MLR_STATUS_CAPACITY);
  }
}

// Per chunk: the stable placement of its pairs.  kBases: the global start of
// every bucket (plus this chunk's earlier-chunk count) is built once in shared
// memory -- for the padded align by scanning the padded bucket totals here
// (which also writes num_tokens_post_pad, the pad sentinels and the block
// labels of this block's share of the buckets: no separate bucket-scan
// launch), for the dense order from dense_start -- so that placing a pair
// reads no global memory.  Without kBases (bucket counts too large for two
// bucket arrays in shared memory) the bases are read per pair from bstart and
// the count matrix, and the pads and labels are written grid-wide.
template <bool kBases>
__global__ void __launch_bounds__(kThreads)
align_scatter_kernel(const int32_t* __restrict__ topk_ids, const int32_t* __restrict__ mapping,
                     int64_t P, int topk, int E, int L, int chunk, int block_size,
                     const uint32_t* __restrict__ cnt, const uint32_t* __restrict__ btotal,
                     const uint32_t* __restrict__ bstart, int32_t* __restrict__ sorted_ids,
                     int32_t* __restrict__ block_expert, int32_t* __restrict__ block_lora,
                     int32_t* __restrict__ num_post_pad, int64_t capacity, int32_t* d_status,
                     const uint32_t* __restrict__ dense_start) {
  pdl_wait();  // the predecessor on the stream has completed
  pdl_trigger();
  // dense_start != nullptr: the dense order (no padding, no labels) for the
  // forward; sorted_ids then receives pair ids at dense_start[b] + rank.
  extern __shared__ uint32_t smem[];
  const int C = L + 1, NB = E * C;
  const int nb4 = (int)round_up(NB + 1, 4);
  // kBases: gb [NB + 1], then off [NB + 1] and stage [chunk], which the final
  // chunk-sorted list (order32 [chunk], one word per pair) later overwrites.
  // Otherwise: off [NB + 1], stage [chunk].
  uint32_t* gb = smem;                                              // (kBases)
  uint32_t* off = smem + (kBases ? nb4 : 0);                        // [NB + 1]
  uint16_t* stage = reinterpret_cast<uint16_t*>(off + nb4);         // [chunk]
  uint32_t* order32 = off;                                          // (kBases) [chunk]
  for (int b = threadIdx.x; b < NB; b += blockDim.x) {
    off[b] = 0u;
    if (kBases) gb[b] = dense_start ? dense_start[b] : (btotal[b] + block_size - 1) / block_size * block_size;
  }
  __syncthreads();

  const int64_t p0 = (int64_t)blockIdx.x * chunk;
  const int n = (int)(P - p0 < chunk ? P - p0 : chunk);
  const int rounds = (n + kThreads - 1) / kThreads;
  // (key << 16) | slot per pair; key < 40960 and slot < 32768 both fit 16 bits.
  // The keys are loaded first (batches of loads in flight), then the counting
  // rounds run on shared memory only.
  uint32_t ks[kMaxItems];
  int bad = 0;
  TokenCursor cur(p0, topk);
#pragma unroll
  for (int bt = 0; bt < kMaxItems; bt += kLoadBatch) {
    int key[kLoadBatch];
    align_load_keys(topk_ids, mapping, p0, n, bt, cur, E, C, L, key, bad);
#pragma unroll
    for (int i = 0; i < kLoadBatch; ++i) ks[bt + i] = key[i] >= 0 ? (uint32_t)key[i] : 0xFFFFFFFFu;
  }
  (void)bad;  // the count kernel reports ids out of range
#pragma unroll
  for (int it = 0; it < kMaxItems; ++it) {
    if (it < rounds) {
      if (ks[it] != 0xFFFFFFFFu) ks[it] = (ks[it] << 16) | atomicAdd(&off[ks[it]], 1u);
      __syncthreads();  // rounds are ordered: a bucket's slots follow round order
    }
  }
  align_block_scan(off, NB);
  const int lane = threadIdx.x & 31;
  const int64_t cap64 = capacity < INT32_MAX ? capacity : INT32_MAX;
  const int cap = (int)cap64, cap_blocks = (int)(cap64 / block_size);
  if (kBases) {
    if (!dense_start) {
      align_block_scan(gb, NB);  // gb[b]: padded start of bucket b; gb[NB]: total
      if (blockIdx.x == 0 && threadIdx.x == 0) {
        *num_post_pad = (int32_t)gb[NB];
        if ((int64_t)gb[NB] > capacity) set_status(d_status, MLR_STATUS_CAPACITY);
      }
      // pad sentinels and block labels of this block's share of the buckets:
      // one warp per bucket, lanes writing consecutive entries
      const int per = (NB + (int)gridDim.x - 1) / (int)gridDim.x;
      const int b0 = min(NB, (int)blockIdx.x * per), b1 = min(NB, b0 + per);
      for (int b = b0 + (threadIdx.x >> 5); b < b1; b += kThreads / 32) {
        const int st = (int)gb[b], en = (int)gb[b + 1];
        if (st == en) continue;
        for (int q = st + (int)btotal[b] + lane; q < en && q < cap; q += 32) sorted_ids[q] = (int32_t)P;
        const int expert = b / C, lora = b - expert * C - 1;
        for (int blk = st / block_size + lane; blk < en / block_size && blk < cap_blocks; blk += 32) {
          block_expert[blk] = expert;
          block_lora[blk] = lora;
        }
      }
      __syncthreads();
    }
    // plus the pairs of each bucket in earlier chunks (coalesced)
    const uint32_t* crow = cnt + (int64_t)blockIdx.x * NB;
    for (int b = threadIdx.x; b < NB; b += blockDim.x) gb[b] += crow[b];
  }
  const int nvalid = (int)off[NB];  // valid pairs of the chunk (off is scanned)
#pragma unroll
  for (int it = 0; it < kMaxItems; ++it)
    if (it < rounds && ks[it] != 0xFFFFFFFFu)
      stage[off[ks[it] >> 16] + (ks[it] & 0xFFFFu)] = (uint16_t)(it * kThreads + threadIdx.x);
  __syncthreads();

  const uint32_t* crow = cnt + (int64_t)blockIdx.x * NB;
#pragma unroll
  for (int it = 0; it < kMaxItems; ++it) {
    if (it < rounds && ks[it] != 0xFFFFFFFFu) {
      const int k = (int)(ks[it] >> 16);
      const uint32_t j = it * kThreads + threadIdx.x;
      const int lo = (int)off[k], hi = (int)off[k + 1];
      const int pos = lo + (int)(ks[it] & 0xFFFFu);
      // same-round neighbours form one contiguous run around pos
      int less = 0, m = pos - 1;
      while (m >= lo && (stage[m] >> 10) == (uint32_t)it) {
        less += stage[m] < j;
        --m;
      }
      const int round_start = m + 1;
      for (m = pos + 1; m < hi && (stage[m] >> 10) == (uint32_t)it; ++m) less += stage[m] < j;
      if (kBases) {
        // the pair's place in the chunk's sorted list (written out below)
        ks[it] = (ks[it] & 0xFFFF0000u) | (uint32_t)(round_start + less);
      } else {
        const int64_t base = (int64_t)(dense_start ? dense_start[k] : bstart[k]) + crow[k];
        const int64_t dst = base + (round_start - lo) + less;
        if (dst < capacity) sorted_ids[dst] = (int32_t)(p0 + j);
      }
    }
  }
  if (kBases) {
    // The chunk's pairs in sorted order in shared memory (over off and stage,
    // which are no longer read), then written out with consecutive threads on
    // consecutive sorted places: the places of one bucket are consecutive in
    // the output too, so the stores coalesce into runs.  gb[k] - off[k] is the
    // output place of the chunk's sorted place 0 for bucket k (gb[k] >= off[k]:
    // the global start of k counts at least this chunk's pairs of earlier buckets).
    __syncthreads();  // every read of off and stage is done
    for (int b = threadIdx.x; b < NB; b += blockDim.x) gb[b] -= off[b];
    __syncthreads();
#pragma unroll
    for (int it = 0; it < kMaxItems; ++it)
      if (it < rounds && ks[it] != 0xFFFFFFFFu)
        order32[ks[it] & 0xFFFFu] = (ks[it] & 0xFFFF0000u) | (uint32_t)(it * kThreads + threadIdx.x);
    __syncthreads();
    for (int q = threadIdx.x; q < nvalid; q += kThreads) {
      const uint32_t v = order32[q];
      const int64_t dst = (int64_t)gb[v >> 16] + q;
      if (dst < capacity) sorted_ids[dst] = (int32_t)(p0 + (v & 0xFFFFu));
    }
    return;
  }
  if (dense_start) return;

  // Pad sentinels and per-block labels: one warp per bucket over the whole
  // grid, lanes writing consecutive entries.  Padded positions are below
  // P + NB * block_size < 2^31 (align_plan checks the bound).
  const int nwarps = gridDim.x * (blockDim.x >> 5);
  for (int b = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); b < NB; b += nwarps) {
    const int st = (int)bstart[b], en = (int)bstart[b + 1];
    if (st == en) continue;
    for (int q = st + (int)btotal[b] + lane; q < en && q < cap; q += 32) sorted_ids[q] = (int32_t)P;
    const int expert = b / C, lora = b - expert * C - 1;
    for (int blk = st / block_size + lane; blk < en / block_size && blk < cap_blocks; blk += 32) {
      block_expert[blk] = expert;
      block_lora[blk] = lora;
    }
  }
}

// Single-block path: the whole align in one launch.
__global__ void __launch_bounds__(kAlignBlockThreads)
align_block_kernel(const int32_t* __restrict__ topk_ids, const int32_t* __restrict__ mapping, int P,
                   int topk, int E, int L, int block_size, int32_t* __restrict__ sorted_ids,
                   int32_t* __restrict__ block_expert, int32_t* __restrict__ block_lora,
                   int32_t* __restrict__ num_post_pad, uint32_t* __restrict__ bstart,
                   int64_t capacity, int32_t* d_status) {
  pdl_wait();  // the predecessor on the stream has completed
  pdl_trigger();
  extern __shared__ __align__(16) unsigned char align_smem[];
  const AlignBlockSmem sm = align_block_carve(align_smem, E * (L + 1), P);
  align_block(topk_ids, mapping, P, topk, E, L, block_size, sm, sorted_ids, block_expert, block_lora,
              num_post_pad, bstart, capacity, d_status);
}

}  // namespace

AlignPlan align_plan(int32_t num_tokens, int32_t topk, int32_t num_experts, int32_t num_loras,
                     int32_t block_size) {
  AlignPlan pl{};
  pl.ok = false;
  if (num_tokens < 0 || topk < 1 || num_experts < 1 || num_loras < 0 || block_size < 1 ||
      block_size > kMaxAlignBlock)
    return pl;
  pl.P = (int64_t)num_tokens * topk;
  const int64_t NB = (int64_t)num_experts * (num_loras + 1);
  if (pl.P >= INT32_MAX || NB > kMaxAlignBuckets) return pl;
  pl.NB = (int)NB;
  // chunks: a whole number of waves of the scatter (one 1024-thread block per
  // SM), each chunk at most kMaxChunk pairs
  const int64_t sms = device_sm_count();
  int64_t chunk = round_up(ceil_div(pl.P, sms), kThreads);
  for (int64_t waves = 2; chunk > kMaxChunk; ++waves) chunk = round_up(ceil_div(pl.P, sms * waves), kThreads);
  chunk = chunk < kThreads ? kThreads : chunk;
  pl.chunk = (int)chunk;
  pl.G = (int)ceil_div(pl.P, chunk);
  const int64_t buckets = pl.P < NB ? pl.P : NB;
  pl.capacity = round_up(pl.P + buckets * (block_size - 1), block_size);
  if (pl.capacity >= INT32_MAX) return pl;
  pl.cnt_off = 0;
  pl.btotal_off = round_up((int64_t)pl.G * NB * 4, 256);
  pl.bstart_off = pl.btotal_off + round_up(NB * 4, 256);
  pl.ws_bytes = pl.bstart_off + round_up((NB + 1) * 4, 256);
  pl.ok = true;
  return pl;
}

size_t align_smem_count(const AlignPlan& pl) { return (size_t)pl.NB * 4; }
// Dynamic shared memory of the scatter: one (or, with the bucket bases, two)
// bucket arrays of round_up(NB + 1, 4) words and the chunk's uint16 stage (with
// the bases, at least 4 bytes per pair of the chunk after the first array).
size_t align_smem_scatter(const AlignPlan& pl, bool bases) {
  const int64_t nb = round_up(pl.NB + 1, 4) * 4, st = round_up((int64_t)pl.chunk * 2, 16);
  if (!bases) return (size_t)(nb + st);
  // gb, then off + stage, which the chunk-sorted list (4 bytes per pair) reuses
  const int64_t tail = nb + st > (int64_t)pl.chunk * 4 ? nb + st : (int64_t)pl.chunk * 4;
  return (size_t)(nb + tail);
}
bool align_bases_fit(const AlignPlan& pl) { return align_smem_scatter(pl, true) <= kSmemLimit; }

template <bool kBases>
int launch_scatter(const AlignPlan& pl, const int32_t* topk_ids, const int32_t* mapping, int topk, int E, int L,
                   int block_size, const uint32_t* cnt, const uint32_t* btotal, const uint32_t* bstart,
                   int32_t* sorted_ids, int32_t* block_expert, int32_t* block_lora, int32_t* num_post_pad,
                   int64_t capacity, int32_t* d_status, const uint32_t* dense_start, cudaStream_t stream) {
  const size_t sm = align_smem_scatter(pl, kBases);
  const int dev = current_device_id();
  static size_t configured[64] = {};  // largest opt-in so far, per device
  if (sm > 48 * 1024 && (dev < 0 || sm > configured[dev])) {
    if (cudaFuncSetAttribute(align_scatter_kernel<kBases>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm) !=
        cudaSuccess)
      return MLR_ERR_CUDA;
    if (dev >= 0) configured[dev] = sm;
  }
  if (launch_pdl(align_scatter_kernel<kBases>, dim3(pl.G), dim3(kThreads), sm, stream, topk_ids, mapping, pl.P, topk, E, L, pl.chunk,
                                                               block_size, cnt, btotal, bstart, sorted_ids,
                                                               block_expert, block_lora, num_post_pad, capacity,
                                                               d_status, dense_start) != cudaSuccess) return MLR_ERR_CUDA;
  MLR_CHECK_LAUNCH();
  note_launch();
  return MLR_OK;
}

int align_launch(const AlignPlan& pl, const int32_t* topk_ids, const int32_t* mapping, int topk,
                 int E, int L, int block_size, int32_t* sorted_ids, int32_t* block_expert,
                 int32_t* block_lora, int32_t* num_post_pad, int64_t capacity, void* workspace,
                 int32_t* d_status, cudaStream_t stream) {
  char* ws = static_cast<char*>(workspace);
  uint32_t* cnt = reinterpret_cast<uint32_t*>(ws + pl.cnt_off);
  uint32_t* btotal = reinterpret_cast<uint32_t*>(ws + pl.btotal_off);
  uint32_t* bstart = reinterpret_cast<uint32_t*>(ws + pl.bstart_off);
  if (align_block_ok(pl)) {
    const size_t sm = align_block_smem(pl);
    if (sm > 48 * 1024 &&
        cudaFuncSetAttribute(align_block_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)sm) != cudaSuccess)
      return MLR_ERR_CUDA;
    if (launch_pdl(align_block_kernel, dim3(1), dim3(kAlignBlockThreads), sm, stream, 
        topk_ids, mapping, (int)pl.P, topk, E, L, block_size, sorted_ids, block_expert, block_lora,
        num_post_pad, bstart, capacity, d_status) != cudaSuccess) return MLR_ERR_CUDA;
    MLR_CHECK_LAUNCH();
    note_launch();
    return MLR_OK;
  }
  const size_t sm_count = align_smem_count(pl);
  if (sm_count > 48 * 1024) {
    if (cudaFuncSetAttribute(align_count_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)sm_count) != cudaSuccess)
      return MLR_ERR_CUDA;
  }
  if (pl.G > 0) {
    if (launch_pdl(align_count_kernel, dim3(pl.G), dim3(kThreads), sm_count, stream, topk_ids, mapping, pl.P, topk, E, L,
                                                             pl.chunk, cnt, d_status) != cudaSuccess) return MLR_ERR_CUDA;
    MLR_CHECK_LAUNCH();
    note_launch();
  }
  if (launch_pdl(align_colscan_kernel, dim3((int)ceil_div(pl.NB, 32)), dim3(kColThreads), 0, stream, cnt, pl.G, pl.NB, btotal) != cudaSuccess) return MLR_ERR_CUDA;
  MLR_CHECK_LAUNCH();
  note_launch();
  if (pl.G > 0 && align_bases_fit(pl))  // the scatter scans the bucket totals itself
    return launch_scatter<true>(pl, topk_ids, mapping, topk, E, L, block_size, cnt, btotal, nullptr, sorted_ids,
                                block_expert, block_lora, num_post_pad, capacity, d_status, nullptr, stream);
  const size_t sm_scan = (size_t)(pl.NB + 1) * 4;
  if (sm_scan > 48 * 1024 &&
      cudaFuncSetAttribute(align_bucketscan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm_scan) !=
          cudaSuccess)
    return MLR_ERR_CUDA;
  if (launch_pdl(align_bucketscan_kernel, dim3(1), dim3(kThreads), sm_scan, stream, btotal, pl.NB, block_size, bstart, num_post_pad,
                                                            capacity, d_status) != cudaSuccess) return MLR_ERR_CUDA;
  MLR_CHECK_LAUNCH();
  note_launch();
  if (pl.G > 0)
    return launch_scatter<false>(pl, topk_ids, mapping, topk, E, L, block_size, cnt, btotal, bstart, sorted_ids,
                                 block_expert, block_lora, num_post_pad, capacity, d_status, nullptr, stream);
  return MLR_OK;
}

int align_dense_count(const AlignPlan& pl, const int32_t* topk_ids, const int32_t* mapping, int topk, int E,
                      int L, void* workspace, int32_t* d_status, cudaStream_t stream) {
  char* ws = static_cast<char*>(workspace);
  uint32_t* cnt = reinterpret_cast<uint32_t*>(ws + pl.cnt_off);
  uint32_t* btotal = reinterpret_cast<uint32_t*>(ws + pl.btotal_off);
  const size_t sm_count = align_smem_count(pl);
  if (sm_count > 48 * 1024 &&
      cudaFuncSetAttribute(align_count_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm_count) !=
          cudaSuccess)
    return MLR_ERR_CUDA;
  if (pl.G > 0) {
    if (launch_pdl(align_count_kernel, dim3(pl.G), dim3(kThreads), sm_count, stream, topk_ids, mapping, pl.P, topk, E, L, pl.chunk, cnt,
                                                             d_status) != cudaSuccess) return MLR_ERR_CUDA;
    MLR_CHECK_LAUNCH();
    note_launch();
  }
  if (launch_pdl(align_colscan_kernel, dim3((int)ceil_div(pl.NB, 32)), dim3(kColThreads), 0, stream, cnt, pl.G, pl.NB, btotal) != cudaSuccess) return MLR_ERR_CUDA;
  MLR_CHECK_LAUNCH();
  note_launch();
  return MLR_OK;
}

int align_dense_scatter(const AlignPlan& pl, const int32_t* topk_ids, const int32_t* mapping, int topk, int E,
                        int L, const void* workspace, const uint32_t* dense_start, int32_t* dense_sorted,
                        cudaStream_t stream) {
  if (pl.G == 0) return MLR_OK;
  const char* ws = static_cast<const char*>(workspace);
  const uint32_t* cnt = reinterpret_cast<const uint32_t*>(ws + pl.cnt_off);
  if (align_bases_fit(pl))
    return launch_scatter<true>(pl, topk_ids, mapping, topk, E, L, 1, cnt, nullptr, nullptr, dense_sorted, nullptr,
                                nullptr, nullptr, pl.P, nullptr, dense_start, stream);
  return launch_scatter<false>(pl, topk_ids, mapping, topk, E, L, 1, cnt, nullptr, nullptr, dense_sorted, nullptr,
                               nullptr, nullptr, pl.P, nullptr, dense_start, stream);
}

}  // namespace mlr

extern "C" int64_t moe_lora_align_capacity(int32_t num_tokens, int32_t topk, int32_t num_experts,
                                           int32_t num_loras, int32_t block_size) {
  const mlr::AlignPlan pl = mlr::align_plan(num_tokens, topk, num_experts, num_loras, block_size);
  return pl.ok ? pl.capacity : -1;
}

extern "C" size_t moe_lora_align_workspace_bytes(int32_t num_tokens, int32_t topk,
                                                 int32_t num_experts, int32_t num_loras,
                                                 int32_t block_size) {
  const mlr::AlignPlan pl = mlr::align_plan(num_tokens, topk, num_experts, num_loras, block_size);
  return pl.ok ? (size_t)pl.ws_bytes : 0;
}

extern "C" int moe_lora_align(const int32_t* topk_ids, const int32_t* token_lora_mapping,
                              int32_t num_tokens, int32_t topk, int32_t num_experts,
                              int32_t num_loras, int32_t block_size, int32_t* sorted_token_ids,
                              int32_t* block_expert_ids, int32_t* block_lora_ids,
                              int32_t* num_tokens_post_pad, int64_t capacity, void* workspace,
                              size_t ws_bytes, int32_t* d_status, void* stream) {
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
  if (workspace == nullptr || ws_bytes < (size_t)pl.ws_bytes) return MLR_ERR_CAPACITY;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255) != 0) return MLR_ERR_INVALID;
  return align_launch(pl, topk_ids, token_lora_mapping, topk, num_experts, num_loras, block_size,
                      sorted_token_ids, block_expert_ids, block_lora_ids, num_tokens_post_pad,
                      capacity, workspace, d_status, static_cast<cudaStream_t>(stream));
}
