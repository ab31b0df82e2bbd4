// forward.cu -- fused_moe_lora_forward: the multi-adapter LoRA MoE expert layer
// (sglang PR #14105 page, 实现拆解: FusedMoEWithLoRA inserts LoRA after the
// gate_up projection and before down; y = (W_down + a/r B_d A_d)[SiLU((W_gate +
// a/r B_g A_g)x) (.) ((W_up + a/r B_u A_u)x)], summed over the top-k experts
// with their routing weights).
//
// Launch sequence (one stream, no host synchronisation):
//   align (block 16)  -> pairs sorted into (expert, adapter) buckets
//   plan              -> tiles: <= 256 consecutive sorted rows of one expert
//                        (base GEMMs) or of one (expert, adapter) bucket (shrinks)
//   shrink_gu         z_gu[row] = s_l * A_gu[l,e] x_t          (gate and up)
//   gate_up           h[row]    = SiLU(W_g x + B_g z_g) * (W_u x + B_u z_u)
//   shrink_d          z_d[row]  = s_l * A_d[l,e] h[row]
//   down              y_acc[t] += w * (W_d h + B_d z_d)
//   convert           y = bf16(y_acc)
// Every GEMM is "swap-AB" on the 5th-generation tensor cores: the weight rows
// are the MMA's M = 128 (A operand), the tile's sorted pair rows are N <= 256
// (B operand), K runs over the hidden / intermediate dimension in 64-wide
// blocks.  Operands are staged in shared memory by TMA (weights, h, LoRA
// factors) or by cp.async gathers (token rows of x), the fp32 accumulator lives
// in TMEM.  Because a tile's rows are sorted by adapter, each adapter owns a
// contiguous column range of the accumulator: the LoRA expand is issued as
// extra MMAs on that column range (N = the bucket's rows) into the same TMEM
// accumulator as the base GEMM, before one epilogue reads it.
#include <cudaTypedefs.h>

#include "mlr_align.cuh"
#include "mlr_profile.cuh"

namespace mlr {
namespace {

constexpr int kBlock = 16;        // internal align block = MMA N granularity
constexpr int kTileRows = 256;    // max sorted rows per tile (MMA N)
constexpr int kMaxBuckets = 20;   // adapter buckets meeting one tile (each >= 16 rows)
constexpr int kMaxExpand = 160;   // expand steps per tile
constexpr int kThreads = 160;     // warps 0-3: producers + epilogue; warp 4: MMA issuer
constexpr int kPlanThreads = 1024;

enum Kind : int { kShrinkGU = 0, kGateUp = 1, kShrinkD = 2, kDown = 3 };

template <int KIND> struct Cfg;
template <> struct Cfg<kShrinkGU> { static constexpr int kStages = 4, kStageBytes = 48 * 1024, kTmemCols = 256; static constexpr bool kGather = true; };
template <> struct Cfg<kGateUp>   { static constexpr int kStages = 3, kStageBytes = 64 * 1024, kTmemCols = 512; static constexpr bool kGather = true; };
template <> struct Cfg<kShrinkD>  { static constexpr int kStages = 4, kStageBytes = 48 * 1024, kTmemCols = 256; static constexpr bool kGather = false; };
template <> struct Cfg<kDown>     { static constexpr int kStages = 4, kStageBytes = 48 * 1024, kTmemCols = 256; static constexpr bool kGather = false; };

struct Maps {
  CUtensorMap m0, m1, m2, m3;
};

struct Params {
  int T, K, E, H, I, L, R, R16, C, mtiles;
  int64_t P;
  const uint16_t* x;
  const float* topk_weights;
  const int32_t* lora_ranks;
  const float* scalings;
  const int32_t* sorted_ids;
  const uint32_t* bstart;  // [E*C + 1] padded bucket starts
  const int4* tiles;       // base: {e, row0, nrows, 0}; shrink: {e, l, row0, nrows}
  const int32_t* n_tiles;
  uint16_t* zgu;  // [cap, 2*R16]
  uint16_t* h;    // [cap, I]
  uint16_t* zd;   // [cap, R16]
  float* yacc;    // [T, H]
  int32_t* status;
};

struct __align__(16) Ctl {
  uint64_t full[4];
  uint64_t empty[4];
  uint64_t accum;
  uint32_t tmem;
  int abort;
  int nb, nexp;
  int bj0[kMaxBuckets], bnj[kMaxBuckets], bl[kMaxBuckets], br16[kMaxBuckets];
  int estep[kMaxExpand];  // bucket << 8 | g << 4 | kg
  int tok[kTileRows];
  float w[kTileRows];
};

template <int KIND>
constexpr int smem_bytes() {
  return Cfg<KIND>::kStages * Cfg<KIND>::kStageBytes + (int)sizeof(Ctl) + 1024;
}

__device__ __forceinline__ float silu_f(float v) { return v / (1.0f + __expf(-v)); }

// Adapter buckets (with a usable LoRA) meeting rows [row0, row0+nrows) of expert e.
__device__ void tile_buckets(const Params& p, int e, int row0, int nrows, int ngates, Ctl& c) {
  const int lo = e * p.C, hi = (e + 1) * p.C;
  int a = lo, b = hi - 1;  // first bucket whose end passes row0
  while (a < b) {
    const int mid = (a + b) >> 1;
    if ((int)p.bstart[mid + 1] > row0) b = mid; else a = mid + 1;
  }
  int nb = 0, ne = 0;
  for (int q = a; q < hi && (int)p.bstart[q] < row0 + nrows; ++q) {
    const int l = q - lo - 1;
    if (l < 0) continue;
    const int r = p.lora_ranks[l];
    if (r < 0 || r > p.R) { set_status(p.status, MLR_STATUS_RANK); continue; }
    if (r == 0) continue;
    const int s0 = max((int)p.bstart[q], row0), s1 = min((int)p.bstart[q + 1], row0 + nrows);
    if (s1 <= s0 || nb >= kMaxBuckets) continue;
    const int r16 = (r + 15) & ~15;
    c.bj0[nb] = s0 - row0; c.bnj[nb] = s1 - s0; c.bl[nb] = l; c.br16[nb] = r16;
    for (int g = 0; g < ngates; ++g)
      for (int kg = 0; kg * 64 < r16; ++kg)
        if (ne < kMaxExpand) c.estep[ne++] = (nb << 8) | (g << 4) | kg;
    ++nb;
  }
  c.nb = nb;
  c.nexp = ne;
}

template <int KIND>
__global__ void __launch_bounds__(kThreads, 1)
moe_gemm_kernel(const __grid_constant__ Maps maps, const Params p) {
  using CF = Cfg<KIND>;
  constexpr int S = CF::kStages;
  constexpr int SB = CF::kStageBytes;
  constexpr bool kShrink = (KIND == kShrinkGU || KIND == kShrinkD);

  // ---- which tile / which M block ----
  const int nblk = kShrink ? p.mtiles : (KIND == kGateUp ? (int)ceil_div(p.I, 128) : (int)ceil_div(p.H, 128));
  const int tile = blockIdx.x / nblk, mb = blockIdx.x % nblk;
  if (tile >= *p.n_tiles) return;
  const int4 td = p.tiles[tile];
  const int e = td.x;
  const int l_shr = kShrink ? td.y : -1;
  const int row0 = kShrink ? td.z : td.y;
  const int nrows = kShrink ? td.w : td.z;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Ctl& c = *reinterpret_cast<Ctl*>(smem + S * SB);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  int r_shr = 0, r16_shr = 0;
  float s_shr = 0.f;
  if (kShrink) {
    r_shr = p.lora_ranks[l_shr];
    r16_shr = (r_shr + 15) & ~15;
    s_shr = p.scalings[l_shr];
  }
  const int nk = (int)ceil_div(KIND == kShrinkGU || KIND == kGateUp ? p.H : p.I, 64);

  // ---- setup ----
  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&c.full[s], CF::kGather ? 129 : 1);
      mbar_init(&c.empty[s], 1);
    }
    mbar_init(&c.accum, 1);
    c.abort = 0;
    c.nb = 0;
    c.nexp = 0;
    if (KIND == kGateUp || KIND == kDown) tile_buckets(p, e, row0, nrows, KIND == kGateUp ? 2 : 1, c);
    fence_mbar_init();
  }
  if (CF::kGather || KIND == kDown) {
    for (int n = tid; n < kTileRows; n += kThreads) {
      const int pr = (n < nrows) ? p.sorted_ids[row0 + n] : (int)p.P;
      const bool real = pr >= 0 && pr < p.P;
      c.tok[n] = real ? pr / p.K : -1;
      if (KIND == kDown) c.w[n] = real ? p.topk_weights[pr] : 0.f;
    }
  }
  if (warp == 4) {
    tmem_alloc(&c.tmem, CF::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = c.tmem;
  const int nsteps = kShrink ? nk : nk + c.nexp;
  volatile int* abort = &c.abort;

  if (warp < 4) {
    // =============================== producer ===============================
    if (CF::kGather || tid == 0) {
      int s = 0;
      for (; s < nsteps; ++s) {
        const int st = s % S, round = s / S;
        uint8_t* sbuf = smem + st * SB;
        if (!mbar_wait(&c.empty[st], (round & 1) ^ 1, abort)) break;
        const bool main_step = s < nk;
        if (tid == 0) {
          if (main_step) {
            const int kb = s;
            if (KIND == kShrinkGU || KIND == kShrinkD) {
              // LoRA A rows packed into M: gate (or the only) rows then up rows, 8-row groups
              int ngr = 0;
              const int r8 = (r_shr + 7) & ~7;
              for (int grp = 0; grp < 16; ++grp) {
                const int m0 = 128 * mb + grp * 8;
                const int g = (KIND == kShrinkGU && m0 >= r16_shr) ? 1 : 0;
                const int q0 = m0 - g * r16_shr;
                if (q0 < r8 && (KIND == kShrinkGU || g == 0)) ++ngr;
              }
              mbar_arrive_expect_tx(&c.full[st], ngr * 1024 + (KIND == kShrinkD ? 32768 : 0));
              for (int grp = 0; grp < 16; ++grp) {
                const int m0 = 128 * mb + grp * 8;
                const int g = (KIND == kShrinkGU && m0 >= r16_shr) ? 1 : 0;
                const int q0 = m0 - g * r16_shr;
                if (!(q0 < r8 && (KIND == kShrinkGU || g == 0))) continue;
                const int row = KIND == kShrinkGU ? ((l_shr * p.E + e) * 2 + g) * p.R + q0
                                                  : (l_shr * p.E + e) * p.R + q0;
                tma_load_2d(sbuf + grp * 1024, &maps.m0, &c.full[st], kb * 64, row);
              }
              if (KIND == kShrinkD) tma_load_2d(sbuf + 16384, &maps.m1, &c.full[st], kb * 64, row0);
            } else if (KIND == kGateUp) {
              mbar_arrive_expect_tx(&c.full[st], 32768);
              const int i0 = mb * 128;
              tma_load_2d(sbuf, &maps.m0, &c.full[st], kb * 64, e * 2 * p.I + i0);
              tma_load_2d(sbuf + 16384, &maps.m0, &c.full[st], kb * 64, e * 2 * p.I + p.I + i0);
            } else {  // kDown
              mbar_arrive_expect_tx(&c.full[st], 16384 + 32768);
              tma_load_2d(sbuf, &maps.m0, &c.full[st], kb * 64, e * p.H + mb * 128);
              tma_load_2d(sbuf + 16384, &maps.m1, &c.full[st], kb * 64, row0);
            }
          } else {
            // expand step: LoRA B chunk (A operand) + z rows of the bucket (B operand)
            const int es = c.estep[s - nk];
            const int bi = es >> 8, g = (es >> 4) & 15, kg = es & 15;
            const int l = c.bl[bi];
            const int nch = min(8, (c.br16[bi] - kg * 64) / 8);
            mbar_arrive_expect_tx(&c.full[st], nch * (2048 + 4096));
            const int m0 = mb * 128;
            const int brow = KIND == kGateUp ? ((l * p.E + e) * 2 + g) * p.I + m0 : (l * p.E + e) * p.H + m0;
            const CUtensorMap* bmap = KIND == kGateUp ? &maps.m1 : &maps.m2;
            const CUtensorMap* zmap = KIND == kGateUp ? &maps.m2 : &maps.m3;
            const int zcol0 = (KIND == kGateUp ? g * p.R16 : 0) + kg * 64;
            for (int ch = 0; ch < nch; ++ch) {
              tma_load_2d(sbuf + ch * 2048, bmap, &c.full[st], kg * 64 + ch * 8, brow);
              tma_load_2d(sbuf + 16384 + ch * 4096, zmap, &c.full[st], zcol0 + ch * 8, row0 + c.bj0[bi]);
            }
          }
        }
        if (CF::kGather) {
          if (main_step) {
            const int kb = s;
            const uint32_t xs = smem_u32(sbuf + (KIND == kGateUp ? 32768 : 16384));
            for (int q = tid; q < nrows * 8; q += 128) {
              const int n = q >> 3, ch = q & 7;
              const int t = c.tok[n];
              const int col = kb * 64 + ch * 8;
              const bool ok = t >= 0 && col < p.H;
              const uint16_t* src = p.x + (ok ? (int64_t)t * p.H + col : 0);
              cp_async_16(xs + n * 128 + ((ch ^ (n & 7)) << 4), src, ok ? 16u : 0u);
            }
          }
          cp_async_commit();
          if (s > 0) {
            cp_async_wait<1>();
            fence_proxy_async_smem();
            mbar_arrive(&c.full[(s - 1) % S]);
          }
        }
      }
      if (CF::kGather && s == nsteps && nsteps > 0) {
        cp_async_wait<0>();
        fence_proxy_async_smem();
        mbar_arrive(&c.full[(nsteps - 1) % S]);
      }
      if (CF::kGather) cp_async_wait<0>();
    }
  } else if (lane == 0) {
    // ================================ MMA ===================================
    for (int s = 0; s < nsteps; ++s) {
      const int st = s % S, round = s / S;
      if (!mbar_wait(&c.full[st], round & 1, abort)) break;
      tc_fence_after();
      const uint32_t sb = smem_u32(smem + st * SB);
      if (s < nk) {
        const uint32_t idesc = idesc_bf16_f32(128, nrows);
        if (KIND == kGateUp) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint32_t acc = (s > 0 || kk > 0) ? 1u : 0u;
            const uint64_t bx = sdesc_sw128(sb + 32768 + kk * 32);
            mma_bf16(tmem, sdesc_sw128(sb + kk * 32), bx, idesc, acc);
            mma_bf16(tmem + 256, sdesc_sw128(sb + 16384 + kk * 32), bx, idesc, acc);
          }
        } else {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_bf16(tmem, sdesc_sw128(sb + kk * 32), sdesc_sw128(sb + 16384 + kk * 32), idesc,
                     (s > 0 || kk > 0) ? 1u : 0u);
        }
      } else {
        const int es = c.estep[s - nk];
        const int bi = es >> 8, g = (es >> 4) & 15, kg = es & 15;
        const int nch = min(8, (c.br16[bi] - kg * 64) / 8);
        const uint32_t d = tmem + (KIND == kGateUp ? g * 256 : 0) + c.bj0[bi];
        const uint32_t idesc = idesc_bf16_f32(128, c.bnj[bi]);
        for (int k16 = 0; k16 < nch / 2; ++k16)
          mma_bf16(d, sdesc_noswz(sb + k16 * 2 * 2048, 2048, 128),
                   sdesc_noswz(sb + 16384 + k16 * 2 * 4096, 4096, 128), idesc, 1u);
      }
      mma_commit(&c.empty[st]);
    }
    mma_commit(&c.accum);
  }

  // ================================ epilogue ================================
  if (warp < 4) {
    const bool ok = mbar_wait(&c.accum, 0, abort);
    tc_fence_after();
    if (ok && !*abort) {
      const uint32_t tl = tmem + ((uint32_t)(warp * 32) << 16);
      const int m = warp * 32 + lane;
      if (KIND == kGateUp) {
        const int gi = mb * 128 + m;
        for (int c0 = 0; c0 < nrows; c0 += 16) {
          float gv[16], uv[16];
          tmem_ld16(tl + c0, gv);
          tmem_ld16(tl + 256 + c0, uv);
          if (gi < p.I) {
#pragma unroll
            for (int j = 0; j < 16; ++j)
              p.h[(int64_t)(row0 + c0 + j) * p.I + gi] = f32_to_bf16_bits(silu_f(gv[j]) * uv[j]);
          }
        }
      } else if (KIND == kDown) {
        const int gh = mb * 128 + m;
        for (int c0 = 0; c0 < nrows; c0 += 16) {
          float v[16];
          tmem_ld16(tl + c0, v);
          if (gh < p.H) {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int t = c.tok[c0 + j];
              if (t >= 0) atomicAdd(p.yacc + (int64_t)t * p.H + gh, c.w[c0 + j] * v[j]);
            }
          }
        }
      } else {
        const int mg = 128 * mb + m;
        int g = 0, q = mg;
        if (KIND == kShrinkGU && mg >= r16_shr) { g = 1; q = mg - r16_shr; }
        const bool valid = KIND == kShrinkGU ? (mg < 2 * r16_shr) : (mg < r16_shr);
        for (int c0 = 0; c0 < nrows; c0 += 16) {
          float v[16];
          tmem_ld16(tl + c0, v);
          if (valid) {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const float z = q < r_shr ? s_shr * v[j] : 0.f;
              if (KIND == kShrinkGU)
                p.zgu[(int64_t)(row0 + c0 + j) * (2 * p.R16) + g * p.R16 + q] = f32_to_bf16_bits(z);
              else
                p.zd[(int64_t)(row0 + c0 + j) * p.R16 + q] = f32_to_bf16_bits(z);
            }
          }
        }
      }
    }
  }
  if (tid == 0 && *abort) set_status(p.status, MLR_STATUS_TIMEOUT);
  tc_fence_before();
  __syncthreads();
  if (warp == 4) tmem_dealloc(tmem, CF::kTmemCols);
}

// Block-wide exclusive scan of per-thread counts; returns this thread's offset.
__device__ int block_offsets(int mine, int* total) {
  __shared__ int wsum[32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int inc = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += v;
  }
  if (lane == 31) wsum[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    const int nw = blockDim.x >> 5;
    int w = lane < nw ? wsum[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += v;
    }
    if (lane < nw) wsum[lane] = w;
  }
  __syncthreads();
  const int off = inc - mine + (warp > 0 ? wsum[warp - 1] : 0);
  *total = wsum[(blockDim.x >> 5) - 1];
  __syncthreads();
  return off;
}

__device__ __forceinline__ void chunk_rows(int n, int k, int nt, int& r0, int& nr) {
  const int cs = (int)round_up(ceil_div(n, nt), kBlock);
  r0 = k * cs;
  nr = min(cs, n - r0);
}

// One block: base tiles per expert and shrink tiles per LoRA bucket.
__global__ void __launch_bounds__(kPlanThreads)
plan_kernel(const uint32_t* __restrict__ bstart, const int32_t* __restrict__ lora_ranks, int E, int C,
            int R, int4* __restrict__ base_tiles, int4* __restrict__ shrink_tiles,
            int32_t* __restrict__ counts, int32_t* status) {
  // base tiles: experts shared out in contiguous ranges
  {
    const int per = (int)ceil_div(E, kPlanThreads);
    const int e0 = min(E, (int)threadIdx.x * per), e1 = min(E, e0 + per);
    int mine = 0;
    for (int e = e0; e < e1; ++e) mine += (int)ceil_div(bstart[(e + 1) * C] - bstart[e * C], kTileRows);
    int total;
    int off = block_offsets(mine, &total);
    for (int e = e0; e < e1; ++e) {
      const int s = (int)bstart[e * C], n = (int)bstart[(e + 1) * C] - s;
      const int nt = (int)ceil_div(n, kTileRows);
      for (int k = 0; k < nt; ++k) {
        int r0, nr;
        chunk_rows(n, k, nt, r0, nr);
        base_tiles[off++] = make_int4(e, s + r0, nr, 0);
      }
    }
    if (threadIdx.x == 0) counts[0] = total;
  }
  // shrink tiles: LoRA buckets (class >= 1, 0 < rank <= R)
  {
    const int NB = E * C;
    const int per = (int)ceil_div(NB, kPlanThreads);
    const int b0 = min(NB, (int)threadIdx.x * per), b1 = min(NB, b0 + per);
    int mine = 0, bad = 0;
    for (int b = b0; b < b1; ++b) {
      const int cl = b % C;
      if (cl == 0) continue;
      const int r = lora_ranks[cl - 1];
      if (r < 0 || r > R) { bad = 1; continue; }
      if (r == 0) continue;
      mine += (int)ceil_div(bstart[b + 1] - bstart[b], kTileRows);
    }
    if (bad) set_status(status, MLR_STATUS_RANK);
    int total;
    int off = block_offsets(mine, &total);
    for (int b = b0; b < b1; ++b) {
      const int cl = b % C;
      if (cl == 0) continue;
      const int r = lora_ranks[cl - 1];
      if (r <= 0 || r > R) continue;
      const int s = (int)bstart[b], n = (int)bstart[b + 1] - s;
      const int nt = (int)ceil_div(n, kTileRows);
      for (int k = 0; k < nt; ++k) {
        int r0, nr;
        chunk_rows(n, k, nt, r0, nr);
        shrink_tiles[off++] = make_int4(b / C, cl - 1, s + r0, nr);
      }
    }
    if (threadIdx.x == 0) counts[1] = total;
  }
}

__global__ void convert_kernel(const float* __restrict__ yacc, uint16_t* __restrict__ y, int64_t n) {
  const int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 4;
  if (i + 4 <= n) {
    const float4 v = *reinterpret_cast<const float4*>(yacc + i);
    uint2 o;
    o.x = (uint32_t)f32_to_bf16_bits(v.x) | ((uint32_t)f32_to_bf16_bits(v.y) << 16);
    o.y = (uint32_t)f32_to_bf16_bits(v.z) | ((uint32_t)f32_to_bf16_bits(v.w) << 16);
    *reinterpret_cast<uint2*>(y + i) = o;
  } else {
    for (int64_t j = i; j < n; ++j) y[j] = f32_to_bf16_bits(yacc[j]);
  }
}

// ----------------------------------------------------------------- host side --
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }
  return fn;
}

// 2-D bf16 tensor [rows, cols] (row-major, row stride = cols) with a box of box_c x box_r.
bool make_map(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint32_t box_c,
              uint32_t box_r, bool swizzle128) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {box_c, box_r};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE,
            swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct FwdLayout {
  bool ok;
  AlignPlan al;
  int R16, C, mtiles_gu, mtiles_d;
  int64_t cap, max_base, max_shrink;
  int64_t o_sorted, o_bexp, o_blora, o_npad, o_align, o_base, o_shrink, o_counts, o_zgu, o_h, o_zd,
      o_yacc, total;
};

FwdLayout fwd_layout(int32_t T, int32_t K, int32_t E, int32_t H, int32_t I, int32_t L, int32_t R) {
  FwdLayout f{};
  f.ok = false;
  if (T < 0 || K < 1 || E < 1 || H < 64 || I < 64 || L < 0 || R < 0) return f;
  if (H % 8 || I % 8 || R % 8 || R > 256 || (L > 0 && R < 8)) return f;
  f.al = align_plan(T, K, E, L, kBlock);
  if (!f.al.ok) return f;
  f.R16 = (int)round_up(R, 16);
  if (f.R16 == 0) f.R16 = 16;
  f.C = L + 1;
  f.mtiles_gu = (int)ceil_div(2 * f.R16, 128);
  f.mtiles_d = (int)ceil_div(f.R16, 128);
  f.cap = f.al.capacity;
  const int64_t nb_nonempty = f.al.P < f.al.NB ? f.al.P : f.al.NB;
  f.max_base = f.cap / kTileRows + E + 1;
  f.max_shrink = f.cap / kTileRows + nb_nonempty + 1;
  int64_t o = 0;
  auto take = [&](int64_t bytes) { const int64_t r = o; o += round_up(bytes > 0 ? bytes : 1, 256); return r; };
  f.o_sorted = take(f.cap * 4);
  f.o_bexp = take(f.cap / kBlock * 4);
  f.o_blora = take(f.cap / kBlock * 4);
  f.o_npad = take(16);
  f.o_align = take(f.al.ws_bytes);
  f.o_base = take(f.max_base * 16);
  f.o_shrink = take(f.max_shrink * 16);
  f.o_counts = take(16);
  f.o_zgu = take(f.cap * 2 * f.R16 * 2);
  f.o_h = take(f.cap * (int64_t)I * 2);
  f.o_zd = take(f.cap * f.R16 * 2);
  f.o_yacc = take((int64_t)T * H * 4);
  f.total = o;
  f.ok = true;
  return f;
}

template <int KIND>
int launch_gemm(const Maps& maps, const Params& p, int64_t max_tiles, int nblk, cudaStream_t stream) {
  const int smem = smem_bytes<KIND>();
  static bool configured = false;
  if (!configured) {
    if (cudaFuncSetAttribute(moe_gemm_kernel<KIND>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
        cudaSuccess)
      return MLR_ERR_CUDA;
    configured = true;
  }
  const int64_t grid = max_tiles * nblk;
  if (grid <= 0) return MLR_OK;
  if (grid > INT32_MAX) return MLR_ERR_UNSUPPORTED;
  moe_gemm_kernel<KIND><<<(unsigned)grid, kThreads, smem, stream>>>(maps, p);
  MLR_CHECK_LAUNCH();
  note_launch();
  return MLR_OK;
}

}  // namespace
}  // namespace mlr

extern "C" size_t fused_moe_lora_workspace_bytes(int32_t num_tokens, int32_t topk, int32_t num_experts,
                                                 int32_t hidden, int32_t intermediate, int32_t num_loras,
                                                 int32_t max_rank) {
  const mlr::FwdLayout f =
      mlr::fwd_layout(num_tokens, topk, num_experts, hidden, intermediate, num_loras, max_rank);
  return f.ok ? (size_t)f.total : 0;
}

extern "C" int fused_moe_lora_forward(const mlr_bf16* x, const int32_t* topk_ids, const float* topk_weights,
                                      const int32_t* token_lora_mapping, const int32_t* lora_ranks,
                                      const float* scalings, const mlr_bf16* w_gate_up,
                                      const mlr_bf16* w_down, const mlr_bf16* lora_a_gu,
                                      const mlr_bf16* lora_b_gu, const mlr_bf16* lora_a_down,
                                      const mlr_bf16* lora_b_down, int32_t T, int32_t K, int32_t E,
                                      int32_t H, int32_t I, int32_t L, int32_t R, mlr_bf16* y,
                                      void* workspace, size_t ws_bytes, int32_t* d_status,
                                      void* stream_) {
  using namespace mlr;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  const FwdLayout f = fwd_layout(T, K, E, H, I, L, R);
  if (!f.ok) {
    if (T < 0 || K < 1 || E < 1 || L < 0 || R < 0) return MLR_ERR_INVALID;
    return MLR_ERR_UNSUPPORTED;
  }
  if (T == 0) return MLR_OK;
  const void* need[] = {x, topk_ids, topk_weights, token_lora_mapping, w_gate_up, w_down, y};
  for (const void* q : need)
    if (q == nullptr) return MLR_ERR_INVALID;
  if (L > 0) {
    const void* lo[] = {lora_ranks, scalings, lora_a_gu, lora_b_gu, lora_a_down, lora_b_down};
    for (const void* q : lo)
      if (q == nullptr) return MLR_ERR_INVALID;
  }
  const void* aligned[] = {x, w_gate_up, w_down, lora_a_gu, lora_b_gu, lora_a_down, lora_b_down, y};
  for (const void* q : aligned)
    if ((reinterpret_cast<uintptr_t>(q) & 15) != 0) return MLR_ERR_INVALID;
  if (workspace == nullptr || ws_bytes < (size_t)f.total) return MLR_ERR_CAPACITY;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255) != 0) return MLR_ERR_INVALID;

  char* ws = static_cast<char*>(workspace);
  int32_t* sorted = reinterpret_cast<int32_t*>(ws + f.o_sorted);
  int32_t* bexp = reinterpret_cast<int32_t*>(ws + f.o_bexp);
  int32_t* blora = reinterpret_cast<int32_t*>(ws + f.o_blora);
  int32_t* npad = reinterpret_cast<int32_t*>(ws + f.o_npad);
  char* aws = ws + f.o_align;
  int4* base_tiles = reinterpret_cast<int4*>(ws + f.o_base);
  int4* shrink_tiles = reinterpret_cast<int4*>(ws + f.o_shrink);
  int32_t* counts = reinterpret_cast<int32_t*>(ws + f.o_counts);
  uint16_t* zgu = reinterpret_cast<uint16_t*>(ws + f.o_zgu);
  uint16_t* hbuf = reinterpret_cast<uint16_t*>(ws + f.o_h);
  uint16_t* zd = reinterpret_cast<uint16_t*>(ws + f.o_zd);
  float* yacc = reinterpret_cast<float*>(ws + f.o_yacc);
  const uint32_t* bstart = reinterpret_cast<const uint32_t*>(aws + f.al.bstart_off);

  // tensor maps
  Maps m_sgu{}, m_gu{}, m_sd{}, m_dn{};
  const uint64_t cap = (uint64_t)f.cap;
  bool ok = make_map(&m_gu.m0, w_gate_up, H, (uint64_t)E * 2 * I, 64, 128, true) &&
            make_map(&m_sd.m1, hbuf, I, cap, 64, 256, true) &&
            make_map(&m_dn.m0, w_down, I, (uint64_t)E * H, 64, 128, true) &&
            make_map(&m_dn.m1, hbuf, I, cap, 64, 256, true);
  if (ok && L > 0) {
    ok = make_map(&m_sgu.m0, lora_a_gu, H, (uint64_t)L * E * 2 * R, 64, 8, true) &&
         make_map(&m_gu.m1, lora_b_gu, R, (uint64_t)L * E * 2 * I, 8, 128, false) &&
         make_map(&m_gu.m2, zgu, 2 * f.R16, cap, 8, 256, false) &&
         make_map(&m_sd.m0, lora_a_down, I, (uint64_t)L * E * R, 64, 8, true) &&
         make_map(&m_dn.m2, lora_b_down, R, (uint64_t)L * E * H, 8, 128, false) &&
         make_map(&m_dn.m3, zd, f.R16, cap, 8, 256, false);
  }
  if (!ok) return MLR_ERR_CUDA;

  const int prof = prof_call_begin(stream);
  if (cudaMemsetAsync(yacc, 0, (size_t)T * H * 4, stream) != cudaSuccess) return MLR_ERR_CUDA;
  int rc = align_launch(f.al, topk_ids, token_lora_mapping, K, E, L, kBlock, sorted, bexp, blora, npad,
                        f.cap, aws, d_status, stream);
  if (rc != MLR_OK) return rc;
  prof_mark(prof, 0, stream);
  plan_kernel<<<1, kPlanThreads, 0, stream>>>(bstart, lora_ranks, E, f.C, R, base_tiles, shrink_tiles,
                                               counts, d_status);
  MLR_CHECK_LAUNCH();
  note_launch();
  prof_mark(prof, 1, stream);

  Params p{};
  p.T = T; p.K = K; p.E = E; p.H = H; p.I = I; p.L = L; p.R = R; p.R16 = f.R16; p.C = f.C;
  p.P = (int64_t)T * K;
  p.x = x;
  p.topk_weights = topk_weights;
  p.lora_ranks = lora_ranks;
  p.scalings = scalings;
  p.sorted_ids = sorted;
  p.bstart = bstart;
  p.zgu = zgu; p.h = hbuf; p.zd = zd; p.yacc = yacc;
  p.status = d_status;

  if (L > 0) {
    Params q = p;
    q.tiles = shrink_tiles; q.n_tiles = counts + 1; q.mtiles = f.mtiles_gu;
    if ((rc = launch_gemm<kShrinkGU>(m_sgu, q, f.max_shrink, f.mtiles_gu, stream)) != MLR_OK) return rc;
  }
  prof_mark(prof, 2, stream);
  {
    Params q = p;
    q.tiles = base_tiles; q.n_tiles = counts; q.mtiles = 1;
    if ((rc = launch_gemm<kGateUp>(m_gu, q, f.max_base, (int)ceil_div(I, 128), stream)) != MLR_OK) return rc;
  }
  prof_mark(prof, 3, stream);
  if (L > 0) {
    Params q = p;
    q.tiles = shrink_tiles; q.n_tiles = counts + 1; q.mtiles = f.mtiles_d;
    if ((rc = launch_gemm<kShrinkD>(m_sd, q, f.max_shrink, f.mtiles_d, stream)) != MLR_OK) return rc;
  }
  prof_mark(prof, 4, stream);
  {
    Params q = p;
    q.tiles = base_tiles; q.n_tiles = counts; q.mtiles = 1;
    if ((rc = launch_gemm<kDown>(m_dn, q, f.max_base, (int)ceil_div(H, 128), stream)) != MLR_OK) return rc;
  }
  prof_mark(prof, 5, stream);
  const int64_t n = (int64_t)T * H;
  convert_kernel<<<(unsigned)ceil_div(ceil_div(n, 4), 256), 256, 0, stream>>>(yacc, y, n);
  MLR_CHECK_LAUNCH();
  note_launch();
  prof_mark(prof, 6, stream);
  return MLR_OK;
}
