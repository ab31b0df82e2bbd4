// forward.cu -- fused_moe_lora_forward: the multi-adapter LoRA MoE expert layer
// (sglang PR #14105 page, 实现拆解: FusedMoEWithLoRA inserts LoRA after the
// gate_up projection and before down; y = (W_down + a/r B_d A_d)[SiLU((W_gate +
// a/r B_g A_g)x) (.) ((W_up + a/r B_u A_u)x)], summed over the top-k experts
// with their routing weights).
//
// Launch sequence (one stream, no host synchronisation):
//   align + plan      pairs sorted stably into (expert, adapter) buckets, in a
//                     dense order (no padding); base tiles (16-aligned, <= 256
//                     rows of one expert, with the LoRA pieces they meet) and
//                     shrink tiles (one bucket's z region); one launch up to
//                     16384 pairs, else counts -> plan -> dense scatter
//   gather_x          x_sorted[u] = x[token of the u-th pair]; y_acc = 0
//   shrink_gu         z_gu[bucket region] = s_l * A_gu[l,e] x_sorted   (gate, up)
//                     (buckets of <= 4 pairs on CUDA cores when buckets are small)
//   gate_up           h[u] = SiLU(W_g x + B_g z_g) * (W_u x + B_u z_u)
//   shrink_d          z_d[bucket region] = s_l * A_d[l,e] h
//   down              y_acc[t] += w * (W_d h + B_d z_d)
//   convert           y = bf16(y_acc)
//
// The four GEMMs share one persistent, warp-specialised kernel on the 5th
// generation tensor cores.  One CTA per SM walks a static share of the work
// items (tile x 128-row weight block).  Every GEMM is "swap-AB": weight rows are
// the MMA's M = 128 (A operand), the tile's sorted pair rows are N <= 256 (B
// operand), K advances in 64-wide blocks through a ring of shared-memory stages
// that keeps streaming across item boundaries:
//   warp 0     producer (lane 0): TMA for weights, LoRA factors and the
//              contiguous row tiles of x_sorted / h / z.  No thread waits for a
//              copy, so every stage of the ring can be in flight.  (Gathering
//              token rows inside the GEMM, 128 bytes per row and K block, moved
//              too few bytes per request; one copy into sorted order first lets
//              every operand load be a large tiled box.)
//   warp 4     TMEM allocation and the single-thread MMA issue (tcgen05.mma)
//   warps 5-   epilogue: TMEM -> registers -> global, overlapping the next
//              item's main loop (double-buffered accumulators where TMEM allows)
// Because a tile's rows are sorted by adapter, each adapter owns a contiguous
// column range of the accumulator: the LoRA expand is issued as extra MMAs on
// that range, rounded out to 16 columns (the z rows outside the bucket are
// zero), into the same TMEM accumulator as the base GEMM, before the epilogue
// reads it.
#include <cudaTypedefs.h>

#include "mlr_align.cuh"
#include "mlr_profile.cuh"

namespace mlr {
namespace {

constexpr int kBlock = 16;        // internal align block = MMA N granularity
constexpr int kTileRows = 256;    // max sorted rows per tile (MMA N)
constexpr int kPlanBigTiles = 8;   // experts with at least this many tiles are planned by the whole block
constexpr int kPlanBigQueue = 64;  // ... up to this many such experts (the rest by their owner thread)
constexpr int kInlinePieces = 30;  // LoRA pieces stored inside a base-tile record
constexpr int kEpiWarp0 = 5;
constexpr int kMaxThreads = 416;  // up to 13 warps (warps 1-3 idle)
constexpr int kGatherThreads = 256;
constexpr int kPlanThreads = 1024;
constexpr int kPlanRankCache = 1024;  // adapters whose ranks the plan keeps in shared memory
constexpr int kShrinkRows = 128;  // max sorted rows per shrink tile
constexpr int kGemvRows = 4;      // buckets with at most this many pairs take the CUDA-core shrink
constexpr int kGemvThreads = 256;
constexpr int kEpiBytes = 32 * (128 + 8) * 2;
constexpr uint64_t kCopyGraceNs = 1000000;  // after an abort: time for issued TMA copies to land  // staging per epilogue half: 32 rows of bf16 h, or 16 rows of fp32

enum Kind : int { kShrinkGU = 0, kGateUp = 1, kShrinkD = 2, kDown = 3 };
// Base expert weight formats: bf16, or codes that converter warps dequantise
// on chip -- FP8 E4M3 and INT8 with 128 x 128 block scales, UINT4 (two per
// byte) with a scale and zero point per row and 128-column group -- or FP8
// E4M3 with power-of-two block scales fed to the FP8 tensor cores as they are
// (kQMx: block-scaled MMAs on E4M3 weights and E4M3-quantised activations).
enum QFmt : int { kQNone = 0, kQFp8 = 1, kQInt8 = 2, kQU4 = 3, kQMx = 4 };
// Formats that go through the converter warps.
template <int QF> constexpr bool kConvOf = QF == kQFp8 || QF == kQInt8 || QF == kQU4;
// Raw code bytes of one weight row per 64-wide K step.
template <int QF> constexpr int kRawRowBytes = QF == kQU4 ? 32 : 64;

// Epilogue warps: the base GEMMs drain their accumulators with two warps per
// TMEM lane quarter, each taking alternate 32-column chunks; the shrinks use
// one warp per quarter.
template <int KIND> constexpr int kEpiWarps = (KIND == kGateUp || KIND == kDown) ? 8 : 4;
template <int KIND> constexpr int kThreadsOf = (kEpiWarp0 + kEpiWarps<KIND>) * 32;
// FP8-weight kernels add three converter warps after the epilogue (16 warps,
// 512 threads): with warps 1-3 they are the six converter warps.
constexpr int kCvWarps = 6;
template <int KIND, int QF> constexpr int kLaunchThreads = kThreadsOf<KIND> + (kConvOf<QF> ? 96 : 0);

template <int KIND> struct Cfg;
// The shrinks stage two 64-wide K chunks per ring slot (LoRA A in [0, 32 KB),
// the x / h rows in [32 KB, 64 KB)): twice the bytes per TMA box.
template <> struct Cfg<kShrinkGU> { static constexpr int kStages = 3, kStageBytes = 64 * 1024, kAccBufs = 2, kAccCols = 256; };
// gate_up (bf16) runs on CTA pairs: a stage holds this CTA's 128-row blocks of
// gate [0, 16 KB) and up [16 KB, 32 KB) and its half of the tile's rows
// [32 KB, 48 KB); the accumulators are gate [0, 256) and up [256, 512).
template <> struct Cfg<kGateUp>   { static constexpr int kStages = 4, kStageBytes = 48 * 1024, kAccBufs = 1, kAccCols = 512; };
template <> struct Cfg<kShrinkD>  { static constexpr int kStages = 3, kStageBytes = 64 * 1024, kAccBufs = 2, kAccCols = 256; };
// down runs on CTA pairs: a stage holds this CTA's 128 weight rows [0, 16 KB)
// and its half of the tile's rows [16 KB, 32 KB).
template <> struct Cfg<kDown>     { static constexpr int kStages = 6, kStageBytes = 32 * 1024, kAccBufs = 2, kAccCols = 256; };

// GEMM kinds that run on CTA pairs (cluster of two, M = 256 tensor-core MMAs):
// each CTA loads half of every row tile, so the row bytes per SM drop by half.
// The bf16 gate_up pair covers 256 rows of I (each CTA its own 128 rows of
// gate and of up, so SiLU(g) * u stays within a CTA) and the bf16 down pair
// 256 rows of H.  The quantised GEMMs run on single CTAs: the converters
// would need a cluster-scope release at every K step, and so would the
// block-scaled MMAs' scale factors (each CTA of a pair reads its own).
template <int KIND, int QF = kQNone> constexpr bool kPairOf = (KIND == kDown || KIND == kGateUp) && QF == kQNone;

// Ring of a GEMM: the FP8 down GEMM on a single CTA stages its 128 weight rows
// [0, 16 KB) and all of the tile's rows [16 KB, 48 KB); the gate_up GEMMs with
// weights dequantised on chip (single CTAs) their gate and up blocks [0, 32 KB)
// and all of the tile's rows [32 KB, 64 KB).
template <int KIND, int QF> struct CfgOf : Cfg<KIND> {};
template <> struct CfgOf<kGateUp, kQFp8> {
  static constexpr int kStages = 3, kStageBytes = 64 * 1024, kAccBufs = 1, kAccCols = 512;
};
template <> struct CfgOf<kGateUp, kQInt8> : CfgOf<kGateUp, kQFp8> {};
template <> struct CfgOf<kGateUp, kQU4> : CfgOf<kGateUp, kQFp8> {};
template <> struct CfgOf<kDown, kQFp8> {
  static constexpr int kStages = 4, kStageBytes = 48 * 1024, kAccBufs = 2, kAccCols = 256;
};
template <> struct CfgOf<kDown, kQInt8> : CfgOf<kDown, kQFp8> {};
template <> struct CfgOf<kDown, kQU4> : CfgOf<kDown, kQFp8> {};
// Block-scaled FP8 (kQMx): a K step is 128 E4M3 codes (128 bytes per row, the
// bf16 kernels' 64 elements), so the stages keep their byte layout.  Tiles
// are at most kMxTileRows rows, which leaves TMEM columns for the scale
// factors after the accumulators: per stage kMxSfCols columns from column
// kAccBufs * kAccCols (A scales of the first [0, 4) and second [4, 8) weight
// block, B scales [8, 16)).  Both GEMMs run on single CTAs with two 128-row
// weight blocks per item sharing the row tile: gate and up for gate_up, two
// consecutive 128-row blocks of W_down for down (which halves the row-tile
// bytes per MMA against one block).  On a CTA pair each CTA's rows read the
// scales in its own TMEM, so the peer's scale-factor writes would have to be
// signalled to the leader at every K step; that per-step signal cost more than
// the pair saved (measured on the down GEMM).
constexpr int kMxTileRows = 224;
constexpr int kMxSfCols = 16;
template <> struct CfgOf<kGateUp, kQMx> {
  static constexpr int kStages = 3, kStageBytes = 64 * 1024, kAccBufs = 1, kAccCols = 2 * kMxTileRows;
};
template <> struct CfgOf<kDown, kQMx> : CfgOf<kGateUp, kQMx> {};
template <int KIND, int QF> constexpr int kSfCol0 = CfgOf<KIND, QF>::kAccBufs * CfgOf<KIND, QF>::kAccCols;
static_assert(kSfCol0<kGateUp, kQMx> + 3 * kMxSfCols <= 512 && kSfCol0<kDown, kQMx> + 4 * kMxSfCols <= 512,
              "scale factors fit TMEM");

// Tensor maps of one GEMM kind, by slot.
//   all:     kW = weight rows (base GEMMs) / LoRA A in 64-row boxes (shrinks),
//            kRows / kRows128 / kRows192 / kRows256 = chunk-major x_sorted or h
//            rows in 64/128/192/256-row boxes (one box = one contiguous run)
//   shrinks: kA32/kA16/kA8 = LoRA A in 32/16/8-row boxes
//            kX2x64 / kX2x128 = x_sorted or h as [chunk][row][64]: one box holds
//            64 or 128 rows of two consecutive 64-wide K chunks
//            kAW16/32/64 ("wide") = LoRA A rows of two K chunks in one box, rb =
//            16/32/64 rank rows (gate_up: [chunk][gate|up][rank][64])
//            kA3x16/kA3x32/kA3x64 (gate_up shrink) = LoRA A viewed as
//            [(l,e,gate|up)][rank][k]: one box holds the gate and up rank rows
//   base:    kB8/kB4/kB2 = LoRA B stack viewed as [rank chunk][row][8 ranks], 8/4/2 chunks per box
//            kZ8/kZ4/kZ2 = chunk-major z viewed the same way, zrows-row boxes;
//            kZ8s/kZ4s/kZ2s the same with 64-row boxes (pieces of <= 64 rows)
//            kW3 (gate_up) = W_gate_up viewed as [(e,gate|up)][row][k]: one
//            box holds a 128-row block of gate and of up
//            kBJ8/kBJ4/kBJ2 (gate_up) = LoRA B viewed as [(l,e,gate|up)][rank
//            chunk][row][8]: one box holds the rank chunks of a gate and of an
//            up block; kZJ4/kZJ2 (zrows-row boxes) and kZJ8s/kZJ4s/kZJ2s
//            (64-row boxes) the z rows of a piece's gate and up columns
// Each TMA box costs the SM's copy engine a roughly fixed time whatever its
// size (measured on GB300 from L2: 8 KB and 32 KB boxes take about the same
// time), so every operand of a K step is fetched with as few boxes as possible.
enum MapSlot {
  kW = 0, kRows = 1, kA32 = 2, kA16 = 3, kA8 = 4, kA3x16 = 5, kA3x32 = 6, kA3x64 = 7,
  kB8 = 2, kB4 = 3, kB2 = 4, kZ8 = 5, kZ4 = 6, kZ2 = 7,
  kX2x64 = 9, kX2x128 = 10, kAW16 = 11, kAW32 = 12, kAW64 = 13,  // shrinks: two-chunk boxes
  kRows128 = 8, kRows256 = 9, kW3 = 10, kZ8s = 11, kZ4s = 12, kZ2s = 13, kRows192 = 14,
  kBJ8 = 15, kBJ4 = 16, kBJ2 = 17, kZJ4 = 18, kZJ2 = 19, kZJ8s = 20, kZJ4s = 21, kZJ2s = 22, kNumMaps = 23,
  kRh32 = 9, kRh96 = 14  // pair kinds: half-tile row boxes of 32 / 96 rows (64 / 128 use kRows / kRows128)
};
struct Maps {
  CUtensorMap m[kNumMaps];
};

// Row space.  The GEMMs work on the dense sorted order: the pairs of every
// (expert, adapter) bucket in align order, buckets back to back with no
// padding (row u of x_sorted / h = the u-th pair).  A LoRA bucket b with dense
// rows [us, ue) owns a z region of rows [floor16(us), ceil16(ue)) in z space,
// starting at z row zstart[b]; its rows outside [us, ue) hold zeros.  An
// expand MMA therefore covers a 16-aligned column range and adds exactly zero
// to the columns of rows outside its bucket.
//
// Base tile: columns [0, N) = dense rows [row0, row0 + N) (row0 16-aligned, N a
// multiple of 16 and <= 256); only columns [lo, hi) belong to expert e.  Its
// LoRA expand work is np pieces {j0 | nj << 16, l, r16, zrow}: the 16-aligned
// column range [j0, j0 + nj) of one bucket, whose z rows start at zrow.  All
// pieces are at pieces[poff..]; the first kInlinePieces are also stored in the
// record so that one warp-wide load brings a whole typical tile.
// gate_up expand: the gate and the up half of a piece share one step when
// both fit a 64 KB stage -- LoRA B of both gates at [0, 32 KB), their z rows
// at [32 KB, 64 KB): pieces of at most 32 ranks (z boxes of up to 256 rows),
// or of 64 ranks over at most 64 columns (z boxes of 64 rows).  The plan
// counts the steps with the same rule.
__host__ __device__ __forceinline__ bool gu_joint_piece(int r16, int nj) {
  return r16 <= 32 || (r16 == 64 && nj <= 64);
}

struct TileRec {
  int4 head;  // {e, row0, N, poff}
  int4 info;  // {lo, hi, np, nexp_gu | nexp_d << 16}: expand steps of gate_up (2 per
              // 64 ranks of a piece, or 1 for a joint piece) and of down (1 per 64 ranks)
  int4 pc[kInlinePieces];
};
static_assert(sizeof(TileRec) == 32 * 16, "one int4 per lane");

// Shrink tile: columns [0, N) = dense rows [row0, row0 + N) of one bucket's z
// region (row0 16-aligned, N <= 128), written to z rows zrow0 + column; bucket
// members are columns [mlo, mhi), the other columns get zeros.
struct ShrinkRec {
  int4 a;  // {e, l, row0, N}
  int4 b;  // {zrow0, mlo, mhi, 0}
};

struct Params {
  int T, K, E, H, I, L, R, R16, C, nblk;
  int cap;    // rows of x_sorted / h per 64-column chunk (dense rows plus slack)
  int zcap;   // rows of z_gu / z_d per 8-column chunk
  int zrows;  // rows per z box (min(256, zcap))
  int zshort; // 1 if the 64-row z maps exist
  int bmask;  // base GEMMs: bit 0 / 1 set if the 8- / 4-chunk LoRA B and z views exist
  int abox_mask;  // shrinks: bit j set if the LoRA A map with (64 >> j)-row boxes exists
  int a3_mask;    // gate_up shrink: bit j set if the gate+up LoRA A map with (16 << j)-row boxes exists
  int aw_mask;    // shrinks: bit j set if the wide LoRA A map with (16 << j)-row boxes exists
  int rmask;      // bit 0 / 1 / 2 set if the 128- / 256- / 192-row maps of the row operand exist
  int ykeep;      // down: 1 if y_acc fits in half of L2 (its reductions are then marked evict-last)
  int zslice_blk; // down: 256-row blocks from this index on read the second rank slice of z (split B)
  int w3;         // gate_up: 1 if the gate+up weight map exists
  int gu_joint;   // gate_up: 1 if the joint gate+up LoRA B and z maps exist (joint expand steps)
  int wsr, wsc;   // FP8 weights: 128-row and 128-column scale blocks per expert matrix
  const float* wscale;  // FP8 / INT8: [E][wsr][wsc] block scales (weight = code x scale);
                        // UINT4: [E][rows][wsc] group scales
  const uint8_t* wzero;   // UINT4: [E][rows][wsc] group zero points
  // block-scaled FP8: weight block exponents [E][wsr][wsc] (scale 2^(e-127)),
  // the B operand's per-row exponents [K/128][cap] (x for gate_up, h for
  // down), and gate_up's outputs: h as E4M3 codes [I/128][cap][128] and its
  // exponents [I/128][cap]
  const uint8_t* wexp;
  const uint8_t* sfx;
  uint8_t* h8;
  uint8_t* sh;
  int64_t P;
  uint64_t wait_ns;  // give-up limit of the pipeline waits
  const float* topk_weights;
  const int32_t* lora_ranks;
  const float* scalings;
  const int32_t* usorted;  // pair id of each dense row
  const TileRec* base_tiles;
  const int4* pieces;
  const ShrinkRec* shrink_tiles;
  const int32_t* n_tiles;
  uint16_t* zgu;  // [2*R16/8][zcap][8]
  uint16_t* h;    // [I/64][cap][64]
  uint16_t* zd;   // [R16/8][zcap][8]
  float* yacc;    // [T, H]
  uint16_t* dpair;  // down, deterministic combine: bf16 w * d of every pair, [P][H] (else null)
  int32_t* status;
};

struct __align__(16) Ctl {
  TileRec rec_p, rec_m;  // the current base tile of the producer / MMA warp
  uint64_t full[8];   // one per ring stage (at most 8)
  uint64_t empty[8];
  uint64_t raw_full[8];  // FP8 weights: the stage's raw weight tile has landed
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint64_t drain;  // pairs: the leader's last commit, waited for before the teardown
  uint32_t tmem;
  int abort;
  int epi_go[2];  // per item parity: one epilogue half may run one item ahead of the other
  int tok[2][kTileRows];  // down: token and top-k weight of each tile column, by item parity
  float w[2][kTileRows];
};

// Block-scaled FP8 gate_up: after Ctl, the column maxima of h that the lane
// quarters of an epilogue half exchange, [half][chunk parity][quarter][32].
template <int KIND, int QF> constexpr int kAmaxBytes = (KIND == kGateUp && QF == kQMx) ? 2 * 2 * 4 * 32 * 4 : 0;

template <int KIND, int QF = kQNone>
constexpr int smem_bytes() {
  using CF = CfgOf<KIND, QF>;
  static_assert(CF::kStages <= 8, "ring barriers");
  return CF::kStages * CF::kStageBytes + (kEpiWarps<KIND> / 4) * kEpiBytes + (int)sizeof(Ctl) +
         kAmaxBytes<KIND, QF> + 1024;
}

// SiLU(v) = v * sigmoid(v), with sigmoid(v) = (1 + tanh(v / 2)) / 2: one
// hardware tanh (tanh.approx.f32, about 2^-11 relative error) and two FMAs,
// half the special-function work of an exponential plus a division.  The
// result is rounded to bf16 right after.  tanh saturates to -1 for v << 0, so
// the product goes to 0, the correct limit.
__device__ __forceinline__ float tanh_approx(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float silu_f(float v) { return v * fmaf(0.5f, tanh_approx(0.5f * v), 0.5f); }
// SiLU to about 1e-6 relative: sigmoid(v) = 1 / (1 + e^-v) with the fast
// exponential and reciprocal (for v << 0, e^-v = inf gives 0, the limit).  The
// block-scaled FP8 layer quantises h to E4M3 right after its bf16 rounding;
// the tanh form's sigmoid loses relative precision for v << 0 (about 0.5% near
// v = -6), enough to move codes across E4M3 rounding boundaries.
__device__ __forceinline__ float silu_acc(float v) { return v * __fdividef(1.f, 1.f + __expf(-v)); }

// One work item: tile rows, weight block, adapter (shrinks: with its rank).
struct Item {
  int e, l, row0, nrows, mb, nexp;
  int np, lo, hi;          // base: LoRA pieces, columns of expert e
  int zrow0, mlo, mhi;     // shrinks: z row of column 0, bucket member columns
  int r, r8, r16;
  int po;   // shrinks: packed M row of the first up rank (gate ranks start at row 0)
  int a3;   // gate_up shrink: rows per gate/up half of the one-box LoRA A load, or 0
  int aw;   // shrinks: rank rows per gate/up half of the wide (two-chunk) A box, or 0
  const int4* pc;          // base: first kInlinePieces pieces (shared or global memory)
  const int4* pg;          // base: all pieces (global memory)
  __device__ __forceinline__ int4 piece(int k) const { return k < kInlinePieces ? pc[k] : pg[k]; }
};

template <int KIND>
__device__ __forceinline__ void item_base(Item& it, const TileRec* rec, const Params& p) {
  const int4 h = rec->head, f = rec->info;
  it.e = h.x; it.l = -1; it.row0 = h.y; it.nrows = h.z;
  it.pg = p.pieces + h.w;
  it.pc = rec->pc;
  it.lo = f.x; it.hi = f.y; it.np = f.z;
  // expand steps: per piece and 64 ranks, one per gate / up for gate_up, one for down
  it.nexp = KIND == kGateUp ? (f.w & 0xffff) : (f.w >> 16);
  it.zrow0 = it.mlo = it.mhi = 0;
  it.r = it.r8 = it.r16 = 0;
  it.po = it.a3 = it.aw = 0;
}

template <int KIND>
__device__ __forceinline__ Item load_item(const Params& p, int item) {
  Item it;
  const int tile = item / p.nblk;
  it.mb = item % p.nblk;
  if (KIND == kShrinkGU || KIND == kShrinkD) {
    const ShrinkRec& t = p.shrink_tiles[tile];
    const int4 a = t.a, b = t.b;
    it.e = a.x; it.l = a.y; it.row0 = a.z; it.nrows = a.w;
    it.zrow0 = b.x; it.mlo = b.y; it.mhi = b.z;
    it.nexp = it.np = it.lo = it.hi = 0;
    it.pc = it.pg = nullptr;
    it.r = p.lora_ranks[it.l];
    it.r8 = (it.r + 7) & ~7;
    it.r16 = (it.r + 15) & ~15;
    it.po = it.r16;
    it.a3 = it.aw = 0;
    if (it.r16 <= 64) {
      const int j = it.r16 <= 16 ? 0 : (it.r16 <= 32 ? 1 : 2);
      if (KIND == kShrinkGU && ((p.a3_mask >> j) & 1)) it.a3 = it.po = 16 << j;
      if ((p.aw_mask >> j) & 1) it.aw = it.po = 16 << j;  // also for the down shrink (po unused there)
    }
  } else {
    item_base<KIND>(it, p.base_tiles + tile, p);
  }
  return it;
}

// load_item for a whole warp: a base tile record (512 bytes) is copied to
// shared memory with one coalesced load and the item reads it from there.  All
// 32 lanes call this.
template <int KIND>
__device__ __forceinline__ Item load_item_warp(const Params& p, int item, TileRec* srec, int lane) {
  if (KIND == kShrinkGU || KIND == kShrinkD) return load_item<KIND>(p, item);
  const int4* src = reinterpret_cast<const int4*>(p.base_tiles + item / p.nblk);
  __syncwarp();  // the previous item's reads of srec are done
  reinterpret_cast<int4*>(srec)[lane] = src[lane];
  __syncwarp();
  Item it;
  it.mb = item % p.nblk;
  item_base<KIND>(it, srec, p);
  return it;
}

// Rows of the z box of an expand piece of nj columns: 64 when the short maps
// exist and suffice, else zrows.
__device__ __forceinline__ int z_box_rows(const Params& p, int nj) { return (nj <= 64 && p.zshort) ? 64 : p.zrows; }

// CTA pairs: rows of this CTA's half of an N-row tile (N a multiple of 16), as
// one box of 32 / 64 / 96 / 128 rows; z rows of half an nj-column piece as one
// box of 64 or 128 rows.
__device__ __forceinline__ int pair_row_box(int nrows) {
  const int h = nrows >> 1;
  return h <= 32 ? 32 : h <= 64 ? 64 : h <= 96 ? 96 : 128;
}
__device__ __forceinline__ int pair_row_slot(int hh) {
  return hh == 32 ? kRh32 : hh == 64 ? kRows : hh == 96 ? kRh96 : kRows128;
}
__device__ __forceinline__ int pair_z_rows(int nj) { return (nj >> 1) <= 64 ? 64 : 128; }

template <bool PAIR>
__device__ __forceinline__ void mma_issue(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  if (PAIR) mma_bf16_pair(d, a, b, idesc, acc);
  else mma_bf16(d, a, b, idesc, acc);
}
// Commit to `bar`; for a pair, to the barrier at the same offset in both CTAs.
template <bool PAIR>
__device__ __forceinline__ void mma_commit_to(uint64_t* bar) {
  if (PAIR) mma_commit_pair(bar, 3);
  else mma_commit(bar);
}

// Bytes between the LoRA A tiles of a shrink stage's two K chunks: the packed
// gate+up (or down) rank rows of the wide / a3 boxes, else a full 128-row M block.
template <int KIND>
__device__ __forceinline__ int shrink_a_stride(const Item& it) {
  const int rb = it.aw ? it.aw : it.a3;
  return rb ? (KIND == kShrinkGU ? 2 : 1) * rb * 128 : 16384;
}

// Walks the expand steps of a base item in order: per bucket, per gate (2 for
// gate_up), per 64 ranks; a joint gate_up step covers both gates of a piece.
// Producer and MMA warp walk the same sequence.
struct ExpandCursor {
  int b = 0, g = 0, kg = 0;
  __device__ __forceinline__ void next(int r16, int ngates, bool joint) {  // r16 of piece b
    if (joint) {
      ++b;
      return;
    }
    if (++kg == (r16 + 63) >> 6) {
      kg = 0;
      if (++g == ngates) {
        g = 0;
        ++b;
      }
    }
  }
};

// Block-scaled FP8: the scale exponents of one main step (K block kb) that a
// lane writes: A exponents of this lane's weight row (gate and up rows for
// gate_up, the rows of both W_down blocks for down), B exponents of tile rows
// 32 i + lane.  Loaded before the stage is free; nothing consumes the loaded
// bytes until sf_store, after the wait, so the loads overlap the wait.
struct SfWords {
  uint32_t a0, a1, b[8];
};
template <int KIND>
__device__ __forceinline__ void sf_load(const Params& p, const Item& it, int kb, int quarter, int lane, SfWords& v) {
  uint32_t e0 = 127u, e1 = 127u;  // rows past I / H read zero codes
  if (KIND == kGateUp) {
    const int r = it.mb * 128 + quarter * 32 + lane;  // row of the gate (and the up) block
    if (r < p.I) {
      e0 = __ldg(p.wexp + ((int64_t)it.e * p.wsr + r / 128) * p.wsc + kb);
      e1 = __ldg(p.wexp + ((int64_t)it.e * p.wsr + (p.I + r) / 128) * p.wsc + kb);
    }
  } else {
    const int r = it.mb * 256 + quarter * 32 + lane;  // row of the first W_down block (second: + 128)
    if (r < p.H) e0 = __ldg(p.wexp + ((int64_t)it.e * p.wsr + r / 128) * p.wsc + kb);
    if (r + 128 < p.H) e1 = __ldg(p.wexp + ((int64_t)it.e * p.wsr + (r + 128) / 128) * p.wsc + kb);
  }
  v.a0 = e0;
  v.a1 = e1;
  const uint8_t* sx = p.sfx + (int64_t)kb * p.cap + it.row0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int n = 32 * i + lane;
    v.b[i] = n < it.nrows ? (uint32_t)__ldg(sx + n) : 127u;
  }
}
// The words into this warp's lane quarter of the stage's scale-factor columns:
// A scales in columns [0, 4) (gate / W_down) and [4, 8) (up) -- the MMA reads
// row m's at column m / 32 of lane m --, B scales of rows 32 i + lane in
// column 8 + i of every quarter.  Every byte of a word holds the same
// exponent, so the four K = 32 MMAs of the step (scale ids 0..3) read the
// same value.
__device__ __forceinline__ void sf_store(uint32_t taddr, const SfWords& v) {
  const uint32_t a0 = v.a0 * 0x01010101u, a1 = v.a1 * 0x01010101u;
  uint32_t w[16] = {a0, a0, a0, a0, a1, a1, a1, a1};
#pragma unroll
  for (int i = 0; i < 8; ++i) w[8 + i] = v.b[i] * 0x01010101u;
  tmem_st16_wait(taddr, w);
}

// Row-box height of a tile of nrows rows (0: several 64-row boxes).
__device__ __forceinline__ int row_box_rows(const Params& p, int nrows) {
  return nrows <= 64 ? 64 : (nrows <= 128 && (p.rmask & 1)) ? 128
                          : (nrows <= 192 && (p.rmask & 4)) ? 192
                          : (nrows <= 256 && (p.rmask & 2)) ? 256 : 0;
}
// Q (gate_up and down only): the expert weights are FP8 E4M3 with 128 x 128
// block scales.  The producer loads the raw codes of a K step into the upper
// half of the stage's weight area; warps 1-3 convert them in place into the
// bf16 tile the MMAs read (code x scale, 128-byte swizzle), so the MMAs, the
// LoRA expand and the epilogue are those of the bf16 kernel.
template <int KIND, int QF = kQNone>
__global__ void __launch_bounds__(kConvOf<QF> ? 512 : kMaxThreads, 1)
moe_gemm_kernel(const __grid_constant__ Maps maps, const Params p) {
  constexpr bool Q = kConvOf<QF>;   // converter warps dequantise the weights
  constexpr bool MX = QF == kQMx;    // block-scaled FP8 MMAs
  static_assert(QF == kQNone || KIND == kGateUp || KIND == kDown, "quantised weights: the base GEMMs only");
  using CF = CfgOf<KIND, QF>;
  constexpr int S = CF::kStages;
  constexpr int SB = CF::kStageBytes;
  constexpr bool kShrink = (KIND == kShrinkGU || KIND == kShrinkD);
  // two weight blocks per item sharing the row tile: gate_up, and the
  // block-scaled down GEMM
  constexpr bool kTwoBlk = KIND == kGateUp || (KIND == kDown && MX);
  // expand units per piece and 64 ranks: gate and up for gate_up; the
  // block-scaled down GEMM expands both of its W_down blocks in one step (they
  // share the piece's z rows, loaded once)
  constexpr int kGates = KIND == kGateUp ? 2 : 1;
  constexpr bool kExp2 = KIND == kDown && MX;
  constexpr int kUOff = MX ? kMxTileRows : 256;  // TMEM column of the second block's accumulator
  // a joint gate_up expand step: LoRA B [0, 32 KB), z rows from 32 KB (at most
  // 32 KB on a single CTA, 16 KB for this CTA's half on a pair)
  static_assert(KIND != kGateUp || SB >= (kPairOf<KIND, QF> ? 48 : 64) * 1024, "joint expand step");
  static_assert(sizeof(Maps) + sizeof(Params) <= 4096, "kernel parameters");

  constexpr bool kPair = kPairOf<KIND, QF>;
  // work unit: a CTA, or for pairs a cluster (both CTAs take the same items and
  // leave together)
  const int unit = kPair ? (int)cluster_id_x() : (int)blockIdx.x;
  const int n_units = kPair ? (int)num_clusters_x() : (int)gridDim.x;
  const uint32_t rank = kPair ? cluster_rank() : 0u;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* epi = smem + S * SB;
  constexpr int kHalves = kEpiWarps<KIND> / 4;  // epilogue warps per TMEM lane quarter
  Ctl& c = *reinterpret_cast<Ctl*>(epi + kHalves * kEpiBytes);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // K steps of 128 bytes per row: 64 bf16 elements, or 128 E4M3 codes for the
  // block-scaled GEMMs
  const int nk = (int)ceil_div(KIND == kShrinkGU || KIND == kGateUp ? p.H : p.I, MX ? 128 : 64);
  const int nks = kShrink ? (nk + 1) / 2 : nk;  // main steps (a shrink step covers two chunks)

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      // FP8: the producer's arrival plus one per converter warp (on a pair,
      // both CTAs' converter warps arrive on the leader's barrier)
      // block-scaled FP8: the producer's expect_tx arrival plus one per
      // scale-factor warp (the producer warp writes lane quarter 0 after
      // issuing the step's copies, warps 1-3 quarters 1-3)
      mbar_init(&c.full[s], Q ? 1 + (kPair ? 2 : 1) * kCvWarps : (MX ? 5 : 1));
      mbar_init(&c.empty[s], 1);
      if (Q) mbar_init(&c.raw_full[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&c.acc_full[b], 1);
      // pairs: one arrival per epilogue half of each CTA, on the leader's barrier
      mbar_init(&c.acc_empty[b], kPair ? 2 * (kEpiWarps<KIND> / 4) : 32 * kEpiWarps<KIND>);
    }
    mbar_init(&c.drain, 1);
    c.abort = 0;
    fence_mbar_init();
  }
  if (warp == 4) {
    if (kPair) {
      tmem_alloc_pair(&c.tmem, 512);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(&c.tmem, 512);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  if (kPair) cluster_sync_all();  // the peer's copies and commits may target this CTA's barriers from here on
  else __syncthreads();
  tc_fence_after();
  // The setup above touches no global memory, so it overlaps the predecessor's
  // last blocks; the plan's outputs are read only after this wait.  A unit
  // without items runs no role's loop and goes straight to the teardown.
  pdl_wait();
  pdl_trigger();
  const int n_items = *p.n_tiles * p.nblk;
  const uint32_t tmem = c.tmem;
  volatile int* abort = &c.abort;

  if (warp == 0) {
    // ================================ producer =================================
    int gs = 0;  // global step counter of this CTA (ring position)
    bool ok = true;
    for (int item = unit; item < n_items && ok; item += n_units) {
      const Item it = load_item_warp<KIND>(p, item, &c.rec_p, lane);
      const int nsteps = nks + it.nexp;
      ExpandCursor cur;
      for (int s = 0; s < nsteps; ++s, ++gs) {
        const int st = gs % S, round = gs / S;
        uint8_t* sbuf = smem + st * SB;
        const bool main_step = s < nks;
        SfWords sfw;
        if (MX && main_step) sf_load<KIND>(p, it, s, 0, lane, sfw);
        const bool w_ok = mbar_wait(&c.empty[st], (round & 1) ^ 1, abort, p.wait_ns);
        if (!__all_sync(0xffffffffu, w_ok)) { ok = false; break; }
        // the row tile of x_sorted / h: one 64/128/192/256-row box where the
        // map exists, else 64-row boxes
        const int hb = row_box_rows(p, it.nrows);
        const int rbox = hb ? 1 : (int)ceil_div(it.nrows, 64);
        const int rbytes = hb ? hb * 128 : rbox * 8192;
        const CUtensorMap* rmap =
            &maps.m[hb == 128 ? kRows128 : hb == 192 ? kRows192 : hb == 256 ? kRows256 : kRows];
        if (lane == 0) {
          if (main_step) {
            const int kb = s;
            if (kShrink) {
              // Two K chunks c0, c0 + 1.  LoRA A rows packed into M: gate rows
              // [0, r8) at packed row 0, up rows at packed row po; chunk kc's A
              // tile starts at kc * ast.  The wide map loads both chunks (and
              // gate and up) in one box; otherwise each chunk is loaded alone,
              // gate+up in one box (a3) or runs of 64/32/16/8-row boxes that
              // never cross a 128-row M-block boundary.
              const int c0 = 2 * kb;
              const int r8 = it.r8, r16 = it.r16;
              const int mlo = 128 * it.mb, mhi = mlo + 128;  // this item's M block
              const int ast = shrink_a_stride<KIND>(it);
              int abytes = 0;
              if (it.aw || it.a3) {
                abytes = it.mb == 0 ? 2 * ast : 0;
              } else {
                for (int g = 0; g < (KIND == kShrinkGU ? 2 : 1); ++g)
                  for (int q = 0; q < r8;) {
                    const int pr = g * r16 + q;
                    int bh = 8;
                    for (int j = 0; j < 4; ++j) {
                      const int cand = 64 >> j;
                      if ((p.abox_mask >> j) & 1 && cand <= r8 - q && (pr >> 7) == ((pr + cand - 1) >> 7)) { bh = cand; break; }
                    }
                    if (pr >= mlo && pr < mhi) abytes += 2 * bh * 128;
                    q += bh;
                  }
              }
              const int xh = it.nrows <= 64 ? 64 : 128;  // x / h rows per chunk
              mbar_arrive_expect_tx(&c.full[st], abytes + 2 * xh * 128);
              if (it.aw) {
                if (it.mb == 0) {
                  const CUtensorMap* am = &maps.m[it.aw == 16 ? kAW16 : it.aw == 32 ? kAW32 : kAW64];
                  if (KIND == kShrinkGU) tma_load_4d(sbuf, am, &c.full[st], 0, 0, (it.l * p.E + it.e) * 2, c0);
                  else tma_load_3d(sbuf, am, &c.full[st], 0, (it.l * p.E + it.e) * p.R, c0);
                }
              } else {
                for (int kc = 0; kc < 2; ++kc) {
                  if (it.a3) {
                    if (it.mb == 0)
                      tma_load_3d(sbuf + kc * ast, &maps.m[it.a3 == 16 ? kA3x16 : it.a3 == 32 ? kA3x32 : kA3x64],
                                  &c.full[st], (c0 + kc) * 64, 0, (it.l * p.E + it.e) * 2);
                    continue;
                  }
                  for (int g = 0; g < (KIND == kShrinkGU ? 2 : 1); ++g)
                    for (int q = 0; q < r8;) {
                      const int pr = g * r16 + q;
                      int bh = 8, bj = 3;
                      for (int j = 0; j < 4; ++j) {
                        const int cand = 64 >> j;
                        if ((p.abox_mask >> j) & 1 && cand <= r8 - q && (pr >> 7) == ((pr + cand - 1) >> 7)) { bh = cand; bj = j; break; }
                      }
                      if (pr >= mlo && pr < mhi) {
                        const int row = KIND == kShrinkGU ? ((it.l * p.E + it.e) * 2 + g) * p.R + q
                                                          : (it.l * p.E + it.e) * p.R + q;
                        const CUtensorMap* am = &maps.m[bj == 0 ? kW : bj == 1 ? kA32 : bj == 2 ? kA16 : kA8];
                        tma_load_2d(sbuf + kc * ast + (pr - mlo) * 128, am, &c.full[st], (c0 + kc) * 64, row);
                      }
                      q += bh;
                    }
                }
              }
              // B operand: rows of x_sorted (gate_up shrink) or h (down shrink), both chunks
              tma_load_3d(sbuf + 32768, &maps.m[xh == 64 ? kX2x64 : kX2x128], &c.full[st], 0, it.row0, c0);
            } else if (KIND == kGateUp) {
              const int i0 = it.mb * 128;
              if (MX) {
                // E4M3 codes of the gate and up blocks, 128 bytes of K per row
                // (the code matrices are mapped as 2-byte elements: the same
                // bytes and swizzle, 64 elements per K step)
                mbar_arrive_expect_tx(&c.full[st], 32768 + rbytes);
                tma_load_3d(sbuf, &maps.m[kW3], &c.full[st], kb * 64, i0, it.e * 2);
              } else if (Q) {
                // raw codes of the gate and up blocks: [gate|up][128 rows][row bytes]
                mbar_arrive_expect_tx(&c.raw_full[st], 256 * kRawRowBytes<QF>);
                tma_load_3d(sbuf + 16384, &maps.m[kW], &c.raw_full[st], kb * kRawRowBytes<QF>, i0, it.e * 2);
                mbar_arrive_expect_tx(&c.full[st], rbytes);
              } else {
                // on the pair: this CTA's 128 rows of the gate and up blocks
                // (rows i0 + 128 rank of the pair's 256) and half of the tile's rows
                const int hh = pair_row_box(it.nrows);
                if (rank == 0) mbar_arrive_expect_tx(&c.full[st], 2 * (32768 + hh * 128));
                const uint32_t fb = cluster_addr(&c.full[st], 0);
                const int ip = it.mb * 256 + (int)rank * 128;
                if (p.w3) {
                  tma_load_3d_pair(sbuf, &maps.m[kW3], fb, kb * 64, ip, it.e * 2);
                } else {
                  tma_load_2d_pair(sbuf, &maps.m[kW], fb, kb * 64, it.e * 2 * p.I + ip);
                  tma_load_2d_pair(sbuf + 16384, &maps.m[kW], fb, kb * 64, it.e * 2 * p.I + p.I + ip);
                }
                tma_load_2d_pair(sbuf + 32768, &maps.m[pair_row_slot(hh)], fb, 0,
                                 kb * p.cap + it.row0 + (int)rank * (it.nrows >> 1));
              }
              if (!kPair)
                for (int q = 0; q < rbox; ++q)
                  tma_load_2d(sbuf + 32768 + q * 8192, rmap, &c.full[st], 0, kb * p.cap + it.row0 + q * 64);
            } else if (!kPair) {
              // kDown with FP8 weights, on a single CTA: raw codes of 128 weight rows
              // on their own barrier, then all of the tile's rows
              static_assert(KIND != kDown || kPair || QF != kQNone, "bf16 down runs on CTA pairs");
              if (MX) {
                // E4M3 codes of two 128-row W_down blocks (one 256-row box),
                // 128 bytes of K per row (mapped as 64 2-byte elements)
                mbar_arrive_expect_tx(&c.full[st], 32768 + rbytes);
                tma_load_2d(sbuf, &maps.m[kW], &c.full[st], kb * 64, it.e * p.H + it.mb * 256);
              } else {
                mbar_arrive_expect_tx(&c.raw_full[st], 128 * kRawRowBytes<QF>);
                tma_load_3d(sbuf + 8192, &maps.m[kW], &c.raw_full[st], kb * kRawRowBytes<QF>, it.mb * 128, it.e);
                mbar_arrive_expect_tx(&c.full[st], rbytes);
              }
              for (int q = 0; q < rbox; ++q)
                tma_load_2d(sbuf + (MX ? 32768 : 16384) + q * 8192, rmap, &c.full[st], 0,
                            kb * p.cap + it.row0 + q * 64);
            } else {  // kDown, on a CTA pair: this CTA's 128 weight rows and half of the tile's rows
              const int hh = pair_row_box(it.nrows);
              if (rank == 0) mbar_arrive_expect_tx(&c.full[st], 2 * (16384 + hh * 128));
              const uint32_t fb = cluster_addr(&c.full[st], 0);
              tma_load_2d_pair(sbuf, &maps.m[kW], fb, kb * 64, it.e * p.H + it.mb * 256 + (int)rank * 128);
              tma_load_2d_pair(sbuf + 16384, &maps.m[pair_row_slot(hh)], fb, 0,
                               kb * p.cap + it.row0 + (int)rank * (it.nrows >> 1));
            }
          } else {
            // expand step: LoRA B chunk (A operand) + z rows of the piece (B operand)
            if (Q) mbar_arrive(&c.raw_full[st]);  // no raw weights: the converters only pass
            const int4 pc = it.piece(cur.b);  // {j0 | nj << 16, l, r16, zrow}
            const int pl = pc.y, pr16 = pc.z, zrow = pc.w;
            const int g = cur.g, kg = cur.kg;
            const bool joint = KIND == kGateUp && p.gu_joint && gu_joint_piece(pr16, pc.x >> 16);
            cur.next(pr16, kGates, joint);
            const int nch = min(8, (pr16 - kg * 64) / 8);  // rank chunks of 8 (even)
            // pairs: this CTA's 128 rows of LoRA B and half of the piece's z rows
            const int zh = kPair ? pair_z_rows(pc.x >> 16) : z_box_rows(p, pc.x >> 16);
            const int zoff = kPair ? (int)rank * ((pc.x >> 16) >> 1) : 0;
            if (joint) {
              // gate and up in one step: LoRA B as [gate|up][chunk][128 rows][8]
              // at [0, 32 KB), z as [gate|up][chunk][zh rows][8] from 32 KB (on a
              // pair: this CTA's 128 rows of B and half of the piece's z rows);
              // 8 chunks come with 64-row z boxes only (gu_joint_piece)
              const int bs = nch == 8 ? kBJ8 : (nch == 4 ? kBJ4 : kBJ2);
              const int zs = zh == 64 ? (nch == 8 ? kZJ8s : (nch == 4 ? kZJ4s : kZJ2s)) : (nch == 4 ? kZJ4 : kZJ2);
              const int bc = (pl * p.E + it.e) * 2;
              if (kPair) {
                if (rank == 0) mbar_arrive_expect_tx(&c.full[st], 2 * 2 * nch * (2048 + zh * 16));
                const uint32_t fb = cluster_addr(&c.full[st], 0);
                tma_load_4d_pair(sbuf, &maps.m[bs], fb, 0, it.mb * 256 + (int)rank * 128, 0, bc);
                tma_load_4d_pair(sbuf + 32768, &maps.m[zs], fb, 0, zrow + zoff, 0, 0);
              } else {
                mbar_arrive_expect_tx(&c.full[st], 2 * nch * (2048 + zh * 16));
                tma_load_4d(sbuf, &maps.m[bs], &c.full[st], 0, it.mb * 128, 0, bc);
                tma_load_4d(sbuf + 32768, &maps.m[zs], &c.full[st], 0, zrow, 0, 0);
              }
            } else {
              // kExp2: LoRA B of both W_down blocks at [0, 16 KB) and [16 KB, 32 KB),
              // the z rows once at [32 KB, 64 KB); else B at [0, 16 KB), z after it
              constexpr int kNb = kExp2 ? 2 : 1;
              const int zbase = kExp2 ? 32768 : 16384;
              if (!kPair) mbar_arrive_expect_tx(&c.full[st], nch * (kNb * 2048 + zh * 16));
              else if (rank == 0) mbar_arrive_expect_tx(&c.full[st], 2 * nch * (2048 + zh * 16));
              const uint32_t fb = kPair ? cluster_addr(&c.full[st], 0) : 0u;
              // z columns of this step: gate_up's gate / up half, or (down with a
              // split B) the rank slice of the output block's part
              const int zslice = (KIND == kDown && it.mb >= p.zslice_blk) ? p.R16 : 0;
              const int zc0 = ((KIND == kGateUp ? g * p.R16 : zslice) + kg * 64) >> 3;
              for (int gb = 0; gb < kNb; ++gb) {
                const int m0 = kPair ? it.mb * 256 + (int)rank * 128 : kExp2 ? it.mb * 256 + gb * 128 : it.mb * 128;
                const int brow = KIND == kGateUp ? ((pl * p.E + it.e) * 2 + g) * p.I + m0
                                                 : (pl * p.E + it.e) * p.H + m0;
                for (int ch = 0; ch < nch;) {
                  const int nc = (nch - ch >= 8 && (p.bmask & 1)) ? 8 : ((nch - ch >= 4 && (p.bmask & 2)) ? 4 : 2);
                  const int bs = nc == 8 ? kB8 : (nc == 4 ? kB4 : kB2);
                  if (kPair) tma_load_3d_pair(sbuf + ch * 2048, &maps.m[bs], fb, 0, brow, kg * 8 + ch);
                  else tma_load_3d(sbuf + gb * 16384 + ch * 2048, &maps.m[bs], &c.full[st], 0, brow, kg * 8 + ch);
                  ch += nc;
                }
              }
              for (int ch = 0; ch < nch;) {
                const int nc = (nch - ch >= 8 && (p.bmask & 1)) ? 8 : ((nch - ch >= 4 && (p.bmask & 2)) ? 4 : 2);
                const int zs = zh == 64 ? (nc == 8 ? kZ8s : (nc == 4 ? kZ4s : kZ2s)) : (nc == 8 ? kZ8 : (nc == 4 ? kZ4 : kZ2));
                if (kPair) tma_load_3d_pair(sbuf + zbase + ch * zh * 16, &maps.m[zs], fb, 0, zrow + zoff, zc0 + ch);
                else tma_load_3d(sbuf + zbase + ch * zh * 16, &maps.m[zs], &c.full[st], 0, zrow, zc0 + ch);
                ch += nc;
              }
            }
          }
        }
        if (MX) {
          // lane quarter 0 of the stage's scale factors, after the copies are
          // issued (the full barrier waits for this arrival too)
          if (main_step) {
            sf_store(tmem + kSfCol0<KIND, QF> + st * kMxSfCols, sfw);
            tc_fence_before();
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&c.full[st]);
        }
      }
    }
  } else if (MX && warp < 4) {
    // ====== block-scaled FP8: scale factors of lane quarters 1-3 (warps 1-3) ======
    // Each main step's A and B scales go into the stage's TMEM columns once
    // the stage is free (the MMAs that read the previous ones have completed),
    // then the warp arrives on the stage's full barrier.
    int gs = 0;
    bool ok = true;
    for (int item = unit; item < n_items && ok; item += n_units) {
      const Item it = load_item<KIND>(p, item);
      const int nsteps = nks + it.nexp;
      for (int s = 0; s < nsteps; ++s, ++gs) {
        const int st = gs % S, round = gs / S;
        SfWords sfw;
        if (s < nks) sf_load<KIND>(p, it, s, warp, lane, sfw);
        const bool w_ok = mbar_wait(&c.empty[st], (round & 1) ^ 1, abort, p.wait_ns);
        if (!__all_sync(0xffffffffu, w_ok)) { ok = false; break; }
        if (s < nks) sf_store(tmem + ((uint32_t)(warp * 32) << 16) + kSfCol0<KIND, QF> + st * kMxSfCols, sfw);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&c.full[st]);
      }
    }
  } else if (Q && (warp < 4 || warp >= kThreadsOf<KIND> / 32)) {
    // ============ converters (quantised weights): raw codes -> bf16 tile ============
    // Warps 1-3 and the three warps after the epilogue.  The raw codes sit in
    // the upper half of the stage's weight area, which the bf16 tile also
    // covers, so every thread first holds its raw chunks in registers and the
    // group meets once (a barrier that also votes on giving up) before anyone
    // writes; then each warp converts its chunks and arrives on its own.  A
    // chunk's scale (and zero point) is fetched before its raw tile is waited for.
    constexpr int kCv = kCvWarps * 32;
    constexpr int kRawOff = KIND == kGateUp ? 16384 : 8192;   // raw codes within the stage
    constexpr int kCpr = kRawRowBytes<QF> / 16;                // 16-byte raw chunks per row
    constexpr int kChunks = (KIND == kGateUp ? 256 : 128) * kCpr;  // raw chunks per K step
    constexpr int kPer = (kChunks + kCv - 1) / kCv;
    const int ct = warp < 4 ? tid - 32 : 96 + tid - kThreadsOf<KIND>;
    int gs = 0;
    for (int item = unit; item < n_items; item += n_units) {
      const Item it = load_item<KIND>(p, item);
      const int nsteps = nks + it.nexp;
      bool stop = false;
      for (int s = 0; s < nsteps; ++s, ++gs) {
        const int st = gs % S, round = gs / S;
        const uint32_t sb = smem_u32(smem + st * SB);
        float scv[kPer], zv[kPer];
        if (s < nks) {
#pragma unroll
          for (int j = 0; j < kPer; ++j) {
            // chunk q = (row ri, chunk of the row); gate_up rows ri = (gate|up, r)
            const int q = ct + kCv * j, ri = q / kCpr;
            const int g = KIND == kGateUp ? (ri >> 7) & 1 : 0;
            const int r = ri & 127;
            const int row = it.mb * 128 + r;  // row of the gate or up matrix, or of W_down
            scv[j] = 0.f;
            zv[j] = 0.f;
            if (q < kChunks && row < (KIND == kGateUp ? p.I : p.H)) {
              const int64_t wrow = KIND == kGateUp ? (int64_t)it.e * 2 * p.I + g * p.I + row
                                                   : (int64_t)it.e * p.H + row;  // row of the stacked matrix
              if (QF == kQU4) {
                const int64_t gi = wrow * p.wsc + (s >> 1);  // this row's 128-column group
                scv[j] = __ldg(p.wscale + gi);
                zv[j] = (float)__ldg(p.wzero + gi);
              } else {
                const int64_t rb = KIND == kGateUp ? (g * p.I + row) / 128 : row / 128;
                scv[j] = __ldg(p.wscale + ((int64_t)it.e * p.wsr + rb) * p.wsc + (s >> 1));
              }
            }
          }
        }
        const bool w_ok = mbar_wait(&c.raw_full[st], round & 1, abort, p.wait_ns);
        uint4 raw[kPer];
        if (s < nks) {
#pragma unroll
          for (int j = 0; j < kPer; ++j) {
            const int q = ct + kCv * j;
            if (q < kChunks) raw[j] = lds128(sb + kRawOff + q * 16);  // (unused if the wait failed)
          }
        }
        // every raw chunk is in registers, and every thread takes the same decision
        if (named_bar_any(4, kCv, !w_ok)) {
          stop = true;
          break;
        }
        if (s < nks) {
#pragma unroll
          for (int j = 0; j < kPer; ++j) {
            const int q = ct + kCv * j;
            if (q >= kChunks) continue;
            const int ri = q / kCpr, c = q % kCpr;
            const int g = KIND == kGateUp ? ri >> 7 : 0;
            const int r = ri & 127;
            const float sc = scv[j];
            const uint32_t rowa = sb + g * 16384 + r * 128;
            if (QF == kQU4) {
              // 32 codes: four words of eight, bf16 units 4c .. 4c + 3 of the row
              const uint32_t wv[4] = {raw[j].x, raw[j].y, raw[j].z, raw[j].w};
#pragma unroll
              for (int v = 0; v < 4; ++v)
                sts128(rowa + (((4 * c + v) ^ (r & 7)) * 16), u4x8_scaled_bf16(wv[v], zv[j], sc));
            } else {
              // 16 codes: bf16 units 2c, 2c + 1 of the row
              uint2 a, b, d, e;
              if (QF == kQFp8) {
                a = e4m3x4_scaled_bf16(raw[j].x, sc);
                b = e4m3x4_scaled_bf16(raw[j].y, sc);
                d = e4m3x4_scaled_bf16(raw[j].z, sc);
                e = e4m3x4_scaled_bf16(raw[j].w, sc);
              } else {
                a = s8x4_scaled_bf16(raw[j].x, sc);
                b = s8x4_scaled_bf16(raw[j].y, sc);
                d = s8x4_scaled_bf16(raw[j].z, sc);
                e = s8x4_scaled_bf16(raw[j].w, sc);
              }
              sts128(rowa + (((2 * c) ^ (r & 7)) * 16), make_uint4(a.x, a.y, b.x, b.y));
              sts128(rowa + (((2 * c + 1) ^ (r & 7)) * 16), make_uint4(d.x, d.y, e.x, e.y));
            }
          }
          fence_proxy_async_smem();  // the tile is read next by the tensor cores
        }
        __syncwarp();  // this warp's chunks are written
        if (lane == 0) {
          if (kPair) mbar_arrive_cluster(cluster_addr(&c.full[st], 0));  // the leader's barrier
          else mbar_arrive(&c.full[st]);
        }
      }
      if (stop) break;
    }
  } else if (warp == 4) {
    // ================== MMA (the warp loads items, one thread issues) ==================
    int gs = 0, il = 0;
    bool ok = true;
    // pairs: the leader issues every MMA; the peer's MMA warp only allocates TMEM
    for (int item = unit; item < n_items && ok && rank == 0; item += n_units, ++il) {
      const Item it = load_item_warp<KIND>(p, item, &c.rec_m, lane);
      if (lane == 0) {
        const int b = il % CF::kAccBufs;
        if (!mbar_wait(&c.acc_empty[b], ((il / CF::kAccBufs) & 1) ^ 1, abort, p.wait_ns)) ok = false;
        tc_fence_after();
        const uint32_t acc = tmem + b * CF::kAccCols;
        const int nsteps = ok ? nks + it.nexp : 0;
        ExpandCursor cur;
        for (int s = 0; s < nsteps; ++s, ++gs) {
          const int st = gs % S, round = gs / S;
          if (!mbar_wait(&c.full[st], round & 1, abort, p.wait_ns)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sb = smem_u32(smem + st * SB);
          if (s < nks && MX) {
            // four K = 32 block-scaled MMAs; scale ids 0..3 pick the (equal) bytes
            const uint32_t sf = tmem + kSfCol0<KIND, QF> + st * kMxSfCols;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint32_t a = (s > 0 || kk > 0) ? 1u : 0u;
              const uint32_t idm = idesc_mx_e4m3(128, it.nrows, kk, kk);
              if (kTwoBlk) {
                const uint64_t bx = sdesc_sw128(sb + 32768 + kk * 32);
                mma_mx(acc, sdesc_sw128(sb + kk * 32), bx, idm, sf, sf + 8, a);
                mma_mx(acc + kUOff, sdesc_sw128(sb + 16384 + kk * 32), bx, idm, sf + 4, sf + 8, a);
              } else {
                mma_mx(acc, sdesc_sw128(sb + kk * 32), sdesc_sw128(sb + 16384 + kk * 32), idm, sf, sf + 8, a);
              }
            }
          } else if (s < nks) {
            const uint32_t idesc = idesc_bf16_f32(kPair ? 256 : 128, it.nrows);
            if (KIND == kGateUp) {
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) {
                const uint32_t a = (s > 0 || kk > 0) ? 1u : 0u;
                const uint64_t bx = sdesc_sw128(sb + 32768 + kk * 32);
                mma_issue<kPair>(acc, sdesc_sw128(sb + kk * 32), bx, idesc, a);
                mma_issue<kPair>(acc + 256, sdesc_sw128(sb + 16384 + kk * 32), bx, idesc, a);
              }
            } else if (kShrink) {
              const int ast = shrink_a_stride<KIND>(it), xst = (it.nrows <= 64 ? 64 : 128) * 128;
#pragma unroll
              for (int kc = 0; kc < 2; ++kc)
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                  mma_issue<kPair>(acc, sdesc_sw128(sb + kc * ast + kk * 32), sdesc_sw128(sb + 32768 + kc * xst + kk * 32),
                           idesc, (s > 0 || kc > 0 || kk > 0) ? 1u : 0u);
            } else {
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                mma_issue<kPair>(acc, sdesc_sw128(sb + kk * 32), sdesc_sw128(sb + 16384 + kk * 32), idesc,
                         (s > 0 || kk > 0) ? 1u : 0u);
            }
          } else {
            const int4 pc = it.piece(cur.b);
            const int g = cur.g, kg = cur.kg;
            const bool joint = KIND == kGateUp && p.gu_joint && gu_joint_piece(pc.z, pc.x >> 16);
            cur.next(pc.z, kGates, joint);
            const int nch = min(8, (pc.z - kg * 64) / 8);
            const int zh = kPair ? pair_z_rows(pc.x >> 16) : z_box_rows(p, pc.x >> 16);
            const uint32_t idesc = idesc_bf16_f32(kPair ? 256 : 128, pc.x >> 16);
            if (joint) {
              // gate and up: LoRA B of gate gg at gg * nch chunks, its z rows at
              // 32 KB + gg * nch chunks of zh rows
              for (int gg = 0; gg < 2; ++gg) {
                const uint32_t d = acc + gg * kUOff + (pc.x & 0xffff);
                const uint32_t bb = sb + gg * nch * 2048, zb = sb + 32768 + gg * nch * zh * 16;
                for (int k16 = 0; k16 < nch / 2; ++k16)
                  mma_issue<kPair>(d, sdesc_noswz(bb + k16 * 2 * 2048, 2048, 128),
                                   sdesc_noswz(zb + k16 * 2 * zh * 16, zh * 16, 128), idesc, 1u);
              }
            } else {
              const uint32_t zb = sb + (kExp2 ? 32768 : 16384);
#pragma unroll
              for (int gb = 0; gb < (kExp2 ? 2 : 1); ++gb) {
                // gate_up: the gate or up accumulator; kExp2: W_down block gb's
                const uint32_t d = acc + (KIND == kGateUp ? g * kUOff : kExp2 ? gb * kUOff : 0) + (pc.x & 0xffff);
                for (int k16 = 0; k16 < nch / 2; ++k16)
                  mma_issue<kPair>(d, sdesc_noswz(sb + gb * 16384 + k16 * 2 * 2048, 2048, 128),
                                   sdesc_noswz(zb + k16 * 2 * zh * 16, zh * 16, 128), idesc, 1u);
              }
            }
          }
          mma_commit_to<kPair>(&c.empty[st]);
        }
        if (ok) mma_commit_to<kPair>(&c.acc_full[b]);
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
    }
    if (kPair && rank == 0 && lane == 0) {
      // the pair's MMAs read both CTAs' shared memory and write both TMEMs:
      // all of them complete before either CTA tears down
      mma_commit_pair(&c.drain, 1);
      if (!mbar_wait_for(&c.drain, 0, kWaitLimitNs)) *abort = 1;
    }
  } else if (warp >= kEpiWarp0) {
    // ================================ epilogue =================================
    const int quarter = warp & 3;  // TMEM lanes this warp may read
    const int m = quarter * 32 + lane;
    const int eh = (warp - kEpiWarp0) >> 2;             // epilogue half (gate_up: 0 or 1)
    const int et = (tid - kEpiWarp0 * 32) & 127;         // 0..127 within the half
    const int ebar = 1 + eh;                             // the half's named barrier (2 halves: 1, 2)
    int il = 0;
    for (int item = unit; item < n_items; item += n_units, ++il) {
      const Item it = load_item<KIND>(p, item);
      const int b = il % CF::kAccBufs;
      if (KIND == kDown) {
        // by item parity: the other half may still read the previous item's
        static_assert(KIND != kDown || kHalves * 128 == kTileRows, "one column per epilogue thread");
        const int n = et + 128 * eh;
        const int pr = (n >= it.lo && n < it.hi) ? p.usorted[it.row0 + n] : (int)p.P;
        const bool real = pr >= 0 && pr < p.P;
        // the token (fp32 reductions into y_acc) or, for the deterministic
        // combine, the pair (its own row of dpair)
        c.tok[il & 1][n] = real ? (p.dpair ? pr : pr / p.K) : -1;
        c.w[il & 1][n] = real ? (p.topk_weights ? p.topk_weights[pr] : 1.f) : 0.f;  // none: weight 1
      }
      // one thread waits for the accumulator; the decision is shared through
      // shared memory so that all 128 epilogue threads take the same branch
      if (et == 0 && eh == 0) {
        const bool got = mbar_wait(&c.acc_full[b], (il / CF::kAccBufs) & 1, abort, p.wait_ns);
        c.epi_go[il & 1] = (got && !*abort) ? 1 : 0;
      }
      if (kHalves == 1) named_bar_sync(1, 128);  // also publishes tok/w
      else named_bar_sync(3, 32 * kEpiWarps<KIND>);
      tc_fence_after();
      if (!c.epi_go[il & 1]) break;
      const uint32_t tl = tmem + b * CF::kAccCols + ((uint32_t)(quarter * 32) << 16);
      if (KIND == kGateUp) {
        // Each warp owns 32 rows of h (its TMEM lane quarter; they lie in one
        // 64-wide chunk of h) and stages 32 columns of them through its own
        // 2 KB of shared memory, then stores 64 contiguous bytes per column.
        // Only the warp synchronises.
        static_assert(KIND != kGateUp || kEpiWarps<KIND> * 2048 <= kHalves * kEpiBytes, "per-warp staging");
        uint16_t* ws = reinterpret_cast<uint16_t*>(epi) + (warp - kEpiWarp0) * 1024;  // [32 columns][32 rows]
        const int iw = (kPair ? it.mb * 256 + (int)rank * 128 : it.mb * 128) + quarter * 32;  // first row of h of this warp
        const bool chunk_ok = iw < (int)round_up(p.I, 64);
        for (int c0 = 32 * eh; c0 < it.nrows; c0 += 32 * kHalves) {  // this half's chunks
          const int ncol = min(32, it.nrows - c0);  // 32 or 16
          if (ncol == 32) {
            float gv[32], uv[32];
            tmem_ld32(tl + c0, gv);
            tmem_ld32(tl + kUOff + c0, uv);
#pragma unroll
            for (int j = 0; j < 32; ++j) ws[j * 32 + lane] = f32_to_bf16_bits((MX ? silu_acc(gv[j]) : silu_f(gv[j])) * uv[j]);
          } else {
            float gv[16], uv[16];
            tmem_ld16(tl + c0, gv);
            tmem_ld16(tl + kUOff + c0, uv);
#pragma unroll
            for (int j = 0; j < 16; ++j) ws[j * 32 + lane] = f32_to_bf16_bits((MX ? silu_acc(gv[j]) : silu_f(gv[j])) * uv[j]);
          }
          __syncwarp();
          // h is chunk-major: [I/64][cap][64]; rows past I are stored as zeros.
          // Only this expert's columns are stored (the others belong to other tiles).
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int q = lane + 32 * k;
            const int n = q >> 2, i = iw + (q & 3) * 8;
            const int col = c0 + n;
            if (n < ncol && chunk_ok && col >= it.lo && col < it.hi) {
              const uint4 v = i < p.I ? *reinterpret_cast<const uint4*>(ws + n * 32 + (q & 3) * 8) : make_uint4(0, 0, 0, 0);
              *reinterpret_cast<uint4*>(p.h + ((int64_t)(i >> 6) * p.cap + it.row0 + col) * 64 + (i & 63)) = v;
            }
          }
          if (MX) {
            // h as E4M3 codes for the block-scaled down GEMM, per column (pair)
            // and the tile's 128 rows of I (one quantisation group): lane j
            // takes column c0 + j, whose 32 rows of this warp are 64 contiguous
            // bytes of the staging area; the half's four lane quarters combine
            // their column maxima through shared memory; each warp writes its
            // 32 codes of the column, quarter 0 also the column's exponent.
            const uint16_t* colp = ws + lane * 32;
            // the column's four pieces of 8 rows, loaded in an order rotated by
            // lane pair so that a warp's loads spread over the banks: ld[r]
            // holds piece (r + rot) & 3, whose codes go to that piece's 8 bytes
            // of the output (the maximum needs no order)
            const int rot = (lane >> 1) & 3;
            uint4 ld[4];
            uint32_t cm2 = 0;  // maxima of |h| bits, two 16-bit halves
#pragma unroll
            for (int r = 0; r < 4; ++r) {
              const int k = (r + rot) & 3;
              ld[r] = *reinterpret_cast<const uint4*>(colp + k * 8);
              if (iw + k * 8 >= p.I) ld[r] = make_uint4(0, 0, 0, 0);  // rows past I (I % 16 == 0)
              cm2 = __vmaxu2(cm2, __vmaxu2(ld[r].x & 0x7fff7fffu, ld[r].y & 0x7fff7fffu));
              cm2 = __vmaxu2(cm2, __vmaxu2(ld[r].z & 0x7fff7fffu, ld[r].w & 0x7fff7fffu));
            }
            const uint32_t cm = max(cm2 & 0xffffu, cm2 >> 16);
            static_assert(!MX || KIND != kGateUp || kAmaxBytes<KIND, QF> == 2048, "column-maxima buffer");
            uint32_t* am = reinterpret_cast<uint32_t*>(reinterpret_cast<uint8_t*>(&c) + sizeof(Ctl)) +
                           (eh * 2 + ((c0 >> 6) & 1)) * 128;
            am[quarter * 32 + lane] = cm;
            named_bar_sync(5 + eh, 128);
            const uint32_t gm = max(max(am[lane], am[32 + lane]), max(am[64 + lane], am[96 + lane]));
            const int sxp = mx_group_exp_bf16(gm);
            const float sc = exp2_neg(sxp);
            const int col = c0 + lane;
            const bool st_ok = lane < ncol && col >= it.lo && col < it.hi;
            uint8_t* dst = p.h8 + ((int64_t)it.mb * p.cap + it.row0 + col) * 128 + quarter * 32;
#pragma unroll
            for (int r = 0; r < 4; ++r) {
              const uint32_t wv[4] = {ld[r].x, ld[r].y, ld[r].z, ld[r].w};
              uint32_t q2[2];
#pragma unroll
              for (int k = 0; k < 4; k += 2) {
                const uint32_t lo = f32x2_to_e4m3x2(__uint_as_float(wv[k] << 16) * sc,
                                                    __uint_as_float(wv[k] & 0xffff0000u) * sc);
                const uint32_t hi = f32x2_to_e4m3x2(__uint_as_float(wv[k + 1] << 16) * sc,
                                                    __uint_as_float(wv[k + 1] & 0xffff0000u) * sc);
                q2[k / 2] = lo | (hi << 16);
              }
              if (st_ok) *reinterpret_cast<uint2*>(dst + ((r + rot) & 3) * 8) = make_uint2(q2[0], q2[1]);
            }
            if (st_ok && quarter == 0) p.sh[(int64_t)it.mb * p.cap + it.row0 + col] = (uint8_t)(sxp + 127);
          }
          __syncwarp();
        }
      } else if (KIND == kDown) {
        // Each warp owns 32 rows of y (its TMEM lane quarter) and transposes
        // 16 columns at a time through its own 2 KB of shared memory, so that a
        // lane then holds 4 consecutive rows of one token: one 16-byte vector
        // reduction into y_acc.  Only the warp synchronises.
        static_assert(KIND != kDown || kEpiWarps<KIND> * 2048 <= kHalves * kEpiBytes, "per-warp staging");
        // two W_down blocks per item (block-scaled FP8): epilogue half eh
        // takes block eh, all columns; otherwise the halves split the columns
        const int hq = (kPair ? it.mb * 256 + (int)rank * 128 : kTwoBlk ? it.mb * 256 + eh * 128 : it.mb * 128) +
                       quarter * 32;
        const uint32_t tlb = tl + (kTwoBlk ? eh * kUOff : 0);
        const int* tk = c.tok[il & 1];
        const float* wk = c.w[il & 1];
        float* wb = reinterpret_cast<float*>(epi) + (warp - kEpiWarp0) * 512;  // [16 columns][32 rows]
        const int q4 = (lane & 7) * 4;   // this lane's 4 rows of y within the warp's 32
        // y_acc rows receive a token's top-k contributions spread over the whole
        // launch; where y_acc fits in half of L2, keep it there against the
        // streamed weights
        const uint64_t ypol = l2_evict_last_policy();
        const bool ykeep = p.ykeep != 0;
        const bool hv = hq + q4 < p.H;   // H is a multiple of 8: all 4 rows or none
        const int cstep = kTwoBlk ? 32 : 32 * kHalves;
        for (int c0 = kTwoBlk ? 0 : 32 * eh; c0 < it.nrows; c0 += cstep) {  // this half's chunks
          const int nc = min(32, it.nrows - c0);  // 32 or 16
          float v[32];
          if (nc == 32) {
            tmem_ld32(tlb + c0, v);
          } else {
            float v16[16];
            tmem_ld16(tlb + c0, v16);
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] = v16[j];
          }
#pragma unroll
          for (int g = 0; g < 32; g += 16) {
            if (g >= nc) break;
#pragma unroll
            for (int j = 0; j < 16; ++j) wb[j * 32 + lane] = v[g + j];
            __syncwarp();
            if (p.dpair) {
              // deterministic combine: a lane holds 8 consecutive rows of one
              // pair and stores w * d as bf16 into the pair's own row (16 B)
#pragma unroll
              for (int k = 0; k < 2; ++k) {
                const int j = k * 8 + (lane >> 2);
                const int n = c0 + g + j;
                const int pr = tk[n];
                const int q8 = (lane & 3) * 8;
                if (hq + q8 < p.H && pr >= 0) {  // H is a multiple of 8: all 8 rows or none
                  const float4 a = *reinterpret_cast<const float4*>(wb + j * 32 + q8);
                  const float4 d = *reinterpret_cast<const float4*>(wb + j * 32 + q8 + 4);
                  const float w = wk[n];
                  uint4 o;
                  o.x = (uint32_t)f32_to_bf16_bits(w * a.x) | ((uint32_t)f32_to_bf16_bits(w * a.y) << 16);
                  o.y = (uint32_t)f32_to_bf16_bits(w * a.z) | ((uint32_t)f32_to_bf16_bits(w * a.w) << 16);
                  o.z = (uint32_t)f32_to_bf16_bits(w * d.x) | ((uint32_t)f32_to_bf16_bits(w * d.y) << 16);
                  o.w = (uint32_t)f32_to_bf16_bits(w * d.z) | ((uint32_t)f32_to_bf16_bits(w * d.w) << 16);
                  *reinterpret_cast<uint4*>(p.dpair + (int64_t)pr * p.H + hq + q8) = o;
                }
              }
              __syncwarp();
              continue;
            }
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const int j = k * 4 + (lane >> 3);  // column of this lane's reduction
              const int n = c0 + g + j;
              const int t = tk[n];
              if (hv && t >= 0) {
                const float4 x = *reinterpret_cast<const float4*>(wb + j * 32 + q4);
                const float w = wk[n];
                float* ya = p.yacc + (int64_t)t * p.H + hq + q4;
                if (ykeep) red_add_v4_hint(ya, w * x.x, w * x.y, w * x.z, w * x.w, ypol);
                else red_add_v4(ya, w * x.x, w * x.y, w * x.z, w * x.w);
              }
            }
            __syncwarp();
          }
        }
      } else {
        const int r = it.r, r16 = it.r16;
        const float sc = p.scalings[it.l];
        const int mg = 128 * it.mb + m;
        int g = 0, q = mg;
        if (KIND == kShrinkGU && mg >= it.po) { g = 1; q = mg - it.po; }
        // rows q in [r16, po) of the gate half hold no rank of this adapter
        const bool valid = q < r16 && (KIND == kShrinkGU ? mg < 2 * it.po : true);
        for (int c0 = 0; c0 < it.nrows; c0 += 16) {
          float v[16];
          tmem_ld16(tl + c0, v);
          if (valid) {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              // columns outside the bucket (and ranks past r) are written as zeros
              const int n = c0 + j;
              const float z = (q < r && n >= it.mlo && n < it.mhi) ? sc * v[j] : 0.f;
              // z is chunk-major: [columns/8][zcap][8]
              const int col = (KIND == kShrinkGU ? g * p.R16 : 0) + q;
              uint16_t* zb = KIND == kShrinkGU ? p.zgu : p.zd;
              zb[((int64_t)(col >> 3) * p.zcap + it.zrow0 + n) * 8 + (col & 7)] = f32_to_bf16_bits(z);
            }
          }
        }
      }
      tc_fence_before();
      named_bar_sync(ebar, 128);  // tok/w and the staging chunk are free for the next item
      if (!kPair) mbar_arrive(&c.acc_empty[b]);
      else if (et == 0) mbar_arrive_cluster(cluster_addr(&c.acc_empty[b], 0));  // the leader's barrier
    }
  }
  if (tid == 0 && *abort) set_status(p.status, MLR_STATUS_TIMEOUT);
  if (*abort) sleep_for_ns(kCopyGraceNs);  // copies already issued land before the teardown
  tc_fence_before();
  if (kPair) cluster_sync_all();  // neither CTA of a pair leaves while the other may still reach it
  else __syncthreads();
  if (warp == 4) {
    if (kPair) tmem_dealloc_pair(tmem, 512);
    else tmem_dealloc(tmem, 512);
  }
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

__device__ __forceinline__ int floor16(int v) { return v & ~15; }
__device__ __forceinline__ int ceil16(int v) { return (v + 15) & ~15; }
// Rows per base tile of an expert spanning `span` rows (a multiple of 16):
// ceil(span / max_rows) tiles of equal size, rounded up to 16 (the count of
// tiles is then ceil(span / tile_rows), every tile non-empty and at most
// max_rows rows; max_rows is 256, or kMxTileRows for the block-scaled FP8
// GEMMs, a multiple of 16 either way).
__device__ __forceinline__ int tile_rows(int span, int max_rows) {
  const int nt = (span + max_rows - 1) / max_rows;
  return ceil16((span + nt - 1) / nt);
}

// One block of kPlanThreads threads.  us[0..NB] (shared memory) holds the dense
// bucket starts (exclusive scan of the bucket sizes, us[NB] = P); zs[0..NB] is
// shared scratch.  Writes the dense starts to ustart_out, the base tiles with
// their LoRA pieces, the shrink tiles (tensor-core and CUDA-core), counts[0] =
// base tiles, counts[1] = tensor-core shrink tiles, counts[2] = CUDA-core ones.
__device__ void plan_block(const uint32_t* us, uint32_t* zs, const int32_t* __restrict__ lora_ranks,
                           int E, int C, int R, uint32_t* __restrict__ ustart_out,
                           TileRec* __restrict__ base_tiles, int4* __restrict__ pieces,
                           ShrinkRec* __restrict__ shrink_tiles, ShrinkRec* __restrict__ gemv_tiles,
                           int32_t* __restrict__ counts, int32_t* status, int gemv_rows, int by_span,
                           int max_rows, int gu_joint) {
  const int NB = E * C;
  int bad = 0;
  // experts with many tiles, planned by the whole block at the end
  __shared__ int big_n;
  __shared__ int4 big_q[kPlanBigQueue];
  if (threadIdx.x == 0) big_n = 0;
  // the adapters' ranks, read once into shared memory when they fit: the
  // per-expert loops below visit every bucket of an expert and would otherwise
  // wait on a global load for each
  __shared__ int32_t rank_cache[kPlanRankCache];
  const int L = C - 1;
  if (L <= kPlanRankCache) {
    for (int l = threadIdx.x; l < L; l += kPlanThreads) rank_cache[l] = lora_ranks[l];
    __syncthreads();
    lora_ranks = rank_cache;
  }
  // z region length of every bucket (LoRA buckets with rank > 0 and pairs only)
  for (int b = threadIdx.x; b < NB; b += kPlanThreads) {
    ustart_out[b] = us[b];
    const int cl = b % C;
    int zl = 0;
    if (cl > 0) {
      const int r = lora_ranks[cl - 1];
      if (r < 0 || r > R) bad = 1;
      else if (r > 0 && us[b + 1] > us[b]) zl = ceil16((int)us[b + 1]) - floor16((int)us[b]);
    }
    zs[b] = (uint32_t)zl;
  }
  if (threadIdx.x == 0) ustart_out[NB] = us[NB];
  __syncthreads();
  align_block_scan(zs, NB);  // zs[b]: first z row of bucket b's region
  // rank rounded to 16 of adapter class cl (adapter cl - 1), 0 for class 0 (no
  // adapter); the per-expert loops walk the classes without a division
  auto rank16c = [&](int cl) -> int {
    if (cl == 0) return 0;
    const int r = lora_ranks[cl - 1];
    return (r > 0 && r <= R) ? (r + 15) & ~15 : 0;
  };
  auto rank16 = [&](int b) -> int { return rank16c(b % C); };  // of bucket b
  // tile k of expert e (tiles of ts rows from r0 over span rows) at slot
  // `slot`, its pieces at pieces[poff ..]; returns the number of pieces
  auto write_tile = [&](int e, int k, int slot, int poff, int r0, int span, int ts) -> int {
    const int ue0 = (int)us[e * C], ue1 = (int)us[(e + 1) * C];
    const int row0 = r0 + k * ts;
    const int N = min(ts, r0 + span - row0);
    TileRec& rec = base_tiles[slot];
    int np = 0, nexp_gu = 0, nexp_d = 0;
    for (int b = e * C + 1, cl = 1; cl < C; ++b, ++cl) {
      const int r16 = rank16c(cl);
      if (r16 == 0 || us[b + 1] == us[b]) continue;
      const int z0 = floor16((int)us[b]), z1 = ceil16((int)us[b + 1]);
      const int a0 = max(z0, row0), a1 = min(z1, row0 + N);
      if (a1 <= a0) continue;
      const int4 pc = make_int4((a0 - row0) | ((a1 - a0) << 16), cl - 1, r16, (int)zs[b] + (a0 - z0));
      pieces[poff + np] = pc;
      if (np < kInlinePieces) rec.pc[np] = pc;
      ++np;
      nexp_gu += (gu_joint && gu_joint_piece(r16, a1 - a0)) ? 1 : 2 * ((r16 + 63) >> 6);
      nexp_d += (r16 + 63) >> 6;
    }
    rec.head = make_int4(e, row0, N, poff);
    rec.info = make_int4(max(ue0, row0) - row0, min(ue1, row0 + N) - row0, np, nexp_gu | (nexp_d << 16));
    return np;
  };
  // ---- base tiles: per expert, equal tiles of <= 256 rows from floor16(first row) ----
  {
    const int per = (E + kPlanThreads - 1) / kPlanThreads;
    const int e0 = min(E, (int)threadIdx.x * per), e1 = min(E, e0 + per);
    int my_t = 0, my_p = 0;
    for (int e = e0; e < e1; ++e) {
      const int ue0 = (int)us[e * C], ue1 = (int)us[(e + 1) * C];
      if (ue1 == ue0) continue;
      const int r0 = floor16(ue0), span = ceil16(ue1) - r0;
      const int ts = tile_rows(span, max_rows), nt = (span + ts - 1) / ts;
      my_t += nt;
      for (int b = e * C + 1, cl = 1; cl < C; ++b, ++cl) {
        if (rank16c(cl) == 0 || us[b + 1] == us[b]) continue;
        if (nt == 1) {  // one tile: every bucket meets it
          ++my_p;
          continue;
        }
        const int z0 = floor16((int)us[b]), z1 = ceil16((int)us[b + 1]);
        my_p += (z1 - 1 - r0) / ts - (z0 - r0) / ts + 1;  // tiles it meets
      }
    }
    int total_t, total_p;
    int toff_seq = block_offsets(my_t, &total_t);  // expert order
    int poff = block_offsets(my_p, &total_p);
    // With by_span, experts are placed in order of decreasing span (64 classes
    // of 16 rows), each expert's tiles in consecutive slots: the static
    // round-robin of items over the CTAs then hands out the largest experts
    // first, while the tiles of one expert still run side by side and share
    // its weights in L2.  The order inside a class follows the shared-memory
    // atomics; no result depends on which CTA runs an item.  Without by_span
    // the experts keep their order (block_offsets above).
    __shared__ int cls_base[64], cls_fill[64];
    auto span_class = [](int span) { return 63 - min(63, span >> 4); };
    if (by_span) {  // uniform over the block
      if (threadIdx.x < 64) {
        cls_base[threadIdx.x] = 0;
        cls_fill[threadIdx.x] = 0;
      }
      __syncthreads();
      for (int e = e0; e < e1; ++e) {
        const int ue0 = (int)us[e * C], ue1 = (int)us[(e + 1) * C];
        if (ue1 == ue0) continue;
        const int span = ceil16(ue1) - floor16(ue0), ts = tile_rows(span, max_rows);
        atomicAdd(&cls_base[span_class(span)], (span + ts - 1) / ts);
      }
      __syncthreads();
      if (threadIdx.x == 0) {
        int run = 0;
        for (int k = 0; k < 64; ++k) {
          const int n = cls_base[k];
          cls_base[k] = run;
          run += n;
        }
      }
      __syncthreads();
    }
    for (int e = e0; e < e1; ++e) {
      const int ue0 = (int)us[e * C], ue1 = (int)us[(e + 1) * C];
      if (ue1 == ue0) continue;
      // nt tiles of equal size (a multiple of 16) over [floor16(first row), ceil16(end))
      const int r0 = floor16(ue0), span = ceil16(ue1) - r0;
      const int ts = tile_rows(span, max_rows), nt = (span + ts - 1) / ts;
      int toff = toff_seq;
      toff_seq += nt;
      if (by_span) {
        const int cls = span_class(span);
        toff = cls_base[cls] + atomicAdd(&cls_fill[cls], nt);
      }
      if (nt >= kPlanBigTiles) {
        // many tiles: queued for the whole block (below); its pieces start at poff
        const int q = atomicAdd(&big_n, 1);
        if (q < kPlanBigQueue) {
          big_q[q] = make_int4(e, toff, poff, 0);
          for (int b = e * C + 1, cl = 1; cl < C; ++b, ++cl) {
            if (rank16c(cl) == 0 || us[b + 1] == us[b]) continue;
            const int z0 = floor16((int)us[b]), z1 = ceil16((int)us[b + 1]);
            poff += (z1 - 1 - r0) / ts - (z0 - r0) / ts + 1;  // tiles it meets
          }
          continue;
        }
      }
      for (int k = 0; k < nt; ++k) poff += write_tile(e, k, toff + k, poff, r0, span, ts);
    }
    if (threadIdx.x == 0) counts[0] = total_t;
  }
  // ---- shrink tiles: each LoRA bucket's z region in pieces of <= 128 rows;
  //      buckets of <= gemv_rows (0 or kGemvRows) pairs go whole to the
  //      CUDA-core shrink ----
  {
    const int per = (NB + kPlanThreads - 1) / kPlanThreads;
    const int b0 = min(NB, (int)threadIdx.x * per), b1 = min(NB, b0 + per);
    int mine = 0, mine_g = 0;
    for (int b = b0; b < b1; ++b) {
      if (rank16(b) == 0 || us[b + 1] == us[b]) continue;
      if ((int)(us[b + 1] - us[b]) <= gemv_rows) ++mine_g;
      else mine += (ceil16((int)us[b + 1]) - floor16((int)us[b]) + kShrinkRows - 1) / kShrinkRows;
    }
    int total, total_g;
    int off = block_offsets(mine, &total);
    int off_g = block_offsets(mine_g, &total_g);
    for (int b = b0; b < b1; ++b) {
      if (rank16(b) == 0 || us[b + 1] == us[b]) continue;
      const int bs = (int)us[b], be = (int)us[b + 1];
      const int z0 = floor16(bs), z1 = ceil16(be);
      const bool small = be - bs <= gemv_rows;  // region of <= 32 rows: one tile
      for (int row0 = z0; row0 < z1; row0 += kShrinkRows) {
        const int N = min(kShrinkRows, z1 - row0);
        ShrinkRec t;
        t.a = make_int4(b / C, b % C - 1, row0, N);
        t.b = make_int4((int)zs[b] + (row0 - z0), max(bs - row0, 0), min(be - row0, N), 0);
        if (small) gemv_tiles[off_g++] = t;
        else shrink_tiles[off++] = t;
      }
    }
    if (threadIdx.x == 0) {
      counts[1] = total;
      counts[2] = total_g;
    }
  }
  {
    // Experts with many tiles: every thread takes tiles of the queued experts.
    // Tile k's pieces start after the pieces of tiles 0..k-1, which is, for
    // each LoRA bucket of the expert (a contiguous run of tiles), the number
    // of its tiles before k.
    const int nbig = min(big_n, kPlanBigQueue);
    for (int qi = 0; qi < nbig; ++qi) {
      const int4 bq = big_q[qi];
      const int e = bq.x;
      const int ue0 = (int)us[e * C], ue1 = (int)us[(e + 1) * C];
      const int r0 = floor16(ue0), span = ceil16(ue1) - r0;
      const int ts = tile_rows(span, max_rows), nt = (span + ts - 1) / ts;
      for (int k = threadIdx.x; k < nt; k += kPlanThreads) {
        int pk = bq.z;
        for (int b = e * C + 1; b < (e + 1) * C; ++b) {
          if (rank16(b) == 0 || us[b + 1] == us[b]) continue;
          const int z0 = floor16((int)us[b]), z1 = ceil16((int)us[b + 1]);
          const int t0 = (z0 - r0) / ts, t1 = (z1 - 1 - r0) / ts;
          pk += max(0, min(t1, k - 1) - t0 + 1);
        }
        write_tile(e, k, bq.y + k, pk, r0, span, ts);
      }
    }
  }
  if (bad) set_status(status, MLR_STATUS_RANK);
}

// Chunked-align path: bucket sizes btotal[NB] -> dense starts, then the plan.
// Dynamic shared memory: 2 * (NB + 1) uint32.
__global__ void __launch_bounds__(kPlanThreads)
plan_kernel(const uint32_t* __restrict__ btotal, const int32_t* __restrict__ lora_ranks, int E, int C,
            int R, uint32_t* __restrict__ ustart, TileRec* __restrict__ base_tiles,
            int4* __restrict__ pieces, ShrinkRec* __restrict__ shrink_tiles,
            ShrinkRec* __restrict__ gemv_tiles, int32_t* __restrict__ counts, int32_t* status,
            int gemv_rows, int by_span, int max_rows, int gu_joint) {
  pdl_wait();  // the predecessor on the stream has completed
  pdl_trigger();
  extern __shared__ __align__(16) unsigned char plan_smem[];
  const int NB = E * C;
  uint32_t* us = reinterpret_cast<uint32_t*>(plan_smem);
  uint32_t* zs = us + round_up(NB + 1, 4);
  for (int b = threadIdx.x; b < NB; b += kPlanThreads) us[b] = btotal[b];
  __syncthreads();
  align_block_scan(us, NB);
  plan_block(us, zs, lora_ranks, E, C, R, ustart, base_tiles, pieces, shrink_tiles, gemv_tiles, counts,
             status, gemv_rows, by_span, max_rows, gu_joint);
}

// Small batches: the single-block align followed by the tile plan, in one
// launch.  The align writes the dense order to usorted and leaves the dense
// bucket starts in its shared count array; the z-region scan uses
// (NB + 1) * 4 more bytes of shared memory at zs_offset.
__global__ void __launch_bounds__(kPlanThreads)
align_plan_kernel(const int32_t* __restrict__ topk_ids, const int32_t* __restrict__ mapping, int P,
                  int topk, int E, int L, int R, const int32_t* __restrict__ lora_ranks,
                  int32_t* __restrict__ usorted, uint32_t* __restrict__ ustart,
                  TileRec* __restrict__ base_tiles, int4* __restrict__ pieces,
                  ShrinkRec* __restrict__ shrink_tiles, ShrinkRec* __restrict__ gemv_tiles,
                  int32_t* __restrict__ counts, int32_t* status, int zs_offset, int gemv_rows, int by_span,
                  int max_rows, int gu_joint) {
  pdl_wait();  // the predecessor on the stream has completed
  pdl_trigger();
  static_assert(kPlanThreads == kAlignBlockThreads, "one block runs both");
  extern __shared__ __align__(16) unsigned char ap_smem[];
  const int C = L + 1, NB = E * C;
  const AlignBlockSmem sm = align_block_carve(ap_smem, NB, P);
  align_block(topk_ids, mapping, P, topk, E, L, kBlock, sm, nullptr, nullptr, nullptr, nullptr, nullptr, P,
              status, usorted);
  plan_block(sm.cnt, reinterpret_cast<uint32_t*>(ap_smem + zs_offset), lora_ranks, E, C, R, ustart,
             base_tiles, pieces, shrink_tiles, gemv_tiles, counts, status, gemv_rows, by_span, max_rows,
             gu_joint);
}

// Dense x_sorted: row u < n = ustart[NB] (the valid pairs) is x[usorted[u] / K]
// (chunk-major [H/64][cap][64], zeros past H); rows [n, cap) are zero.  One
// warp per row, 16-byte loads and stores.  The same launch zeroes y_acc.
__global__ void __launch_bounds__(kGatherThreads)
gather_x_kernel(const uint16_t* __restrict__ x, const int32_t* __restrict__ usorted,
                const uint32_t* __restrict__ n_valid, int K, int H, int64_t cap, uint16_t* __restrict__ xs,
                float* __restrict__ yacc, int64_t yacc_n4) {
  pdl_wait();  // the predecessor on the stream has completed
  pdl_trigger();
  const int64_t n = *n_valid;
  const int lane = threadIdx.x & 31;
  const int64_t wpb = kGatherThreads / 32;
  const int pieces16 = (int)round_up(H, 64) / 8;  // 16-byte pieces per padded row
  const int64_t w0 = (int64_t)blockIdx.x * wpb + (threadIdx.x >> 5), ws = (int64_t)gridDim.x * wpb;
  constexpr int kBatch = 8;  // 16-byte loads in flight per lane (4 KB per warp)
  for (int64_t u = w0; u < cap; u += ws) {
    const bool real = u < n;
    const uint4* src = reinterpret_cast<const uint4*>(x + (real ? (int64_t)(usorted[u] / K) * H : 0));
    for (int c0 = lane; c0 < pieces16; c0 += 32 * kBatch) {
      uint4 v[kBatch];
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        const int c = c0 + 32 * j;
        v[j] = (real && c < pieces16 && c * 8 < H) ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        const int c = c0 + 32 * j;
        if (c < pieces16) *reinterpret_cast<uint4*>(xs + ((int64_t)(c >> 3) * cap + u) * 64 + (c & 7) * 8) = v[j];
      }
    }
  }
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < yacc_n4; i += (int64_t)gridDim.x * blockDim.x)
    reinterpret_cast<float4*>(yacc)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// Position of each placed pair in the dense order: pos[usorted[u]] = u for
// u < n.  Pairs the align leaves out (ids out of range, which it reports)
// are not written; the token-major gathers skip them by the align's own rule.
__global__ void __launch_bounds__(kGatherThreads)
dense_pos_kernel(const int32_t* __restrict__ usorted, const uint32_t* __restrict__ n_valid,
                 int32_t* __restrict__ pos) {
  pdl_wait();  // the predecessor on the stream has completed
  pdl_trigger();
  const int64_t n = *n_valid;
  for (int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; u < n; u += (int64_t)gridDim.x * blockDim.x)
    pos[usorted[u]] = (int32_t)u;
}

// Tasks of the gathers.  Token-major (pos given): task t < T nkc (nkc =
// ceil(K / 32)) is token t / nkc with its pairs k in [32 (t % nkc), + 32),
// whose row of x is read once and written to the dense rows of those pairs
// that the align places (expert in [0, E), adapter in [-1, L)); task T nkc + i
// is the padding row n + i, written as zeros.  Row-major (pos null): task u <
// cap is dense row u, the row of x of pair usorted[u] for u < n, else zeros.
// Lane j returns the task's j-th destination row, or -1; tok is the token
// whose row is read, or -1.
__device__ __forceinline__ int64_t gather_tasks(int T, int K, int64_t n, int64_t cap, const int32_t* pos) {
  return pos ? (int64_t)T * ((K + 31) >> 5) + (cap - n) : cap;
}
__device__ __forceinline__ int gather_task_row(int64_t task, int T, int K, int E, int L, int64_t n,
                                               const int32_t* __restrict__ topk_ids,
                                               const int32_t* __restrict__ mapping,
                                               const int32_t* __restrict__ usorted,
                                               const int32_t* __restrict__ pos, int lane, int64_t& tok) {
  if (pos == nullptr) {
    tok = task < n ? usorted[task] / K : -1;
    return lane == 0 ? (int)task : -1;
  }
  const int nkc = (K + 31) >> 5;
  int u = -1;
  if (task < (int64_t)T * nkc) {
    tok = task / nkc;
    const int k = (int)(task - tok * nkc) * 32 + lane;
    if (k < K) {
      const int64_t pr = tok * K + k;
      const int e = __ldg(topk_ids + pr), l = __ldg(mapping + tok);
      if (e >= 0 && e < E && l >= -1 && l < L) {
        const int v = pos[pr];
        if (v >= 0 && v < n) u = v;  // (a stale entry after a reported index error stays in range)
      }
    }
  } else {
    tok = -1;
    if (lane == 0) u = (int)(n + (task - (int64_t)T * nkc));
  }
  return u;
}

// gather_x_kernel's result (x_sorted [H/64][cap][64], zeros past H and in
// rows [n, cap); y_acc zeroed), token-major: each token's row read once for
// its K pairs.
__global__ void __launch_bounds__(kGatherThreads)
gather_x_tok_kernel(const uint16_t* __restrict__ x, const int32_t* __restrict__ topk_ids,
                    const int32_t* __restrict__ mapping, const int32_t* __restrict__ usorted,
                    const int32_t* __restrict__ pos,
                    const uint32_t* __restrict__ n_valid, int T, int K, int E, int L, int H, int64_t cap,
                    uint16_t* __restrict__ xs, float* __restrict__ yacc, int64_t yacc_n4) {
  pdl_wait();  // the predecessor on the stream has completed
  pdl_trigger();
  const int64_t n = *n_valid;
  const int64_t n_tasks = gather_tasks(T, K, n, cap, pos);
  const int lane = threadIdx.x & 31;
  const int64_t wpb = kGatherThreads / 32;
  const int pieces16 = (int)round_up(H, 64) / 8;  // 16-byte pieces per padded row
  const int64_t w0 = (int64_t)blockIdx.x * wpb + (threadIdx.x >> 5), ws = (int64_t)gridDim.x * wpb;
  constexpr int kBatch = 8;  // 16-byte loads in flight per lane (4 KB per warp)
  for (int64_t task = w0; task < n_tasks; task += ws) {
    int64_t tok;
    const int myu = gather_task_row(task, T, K, E, L, n, topk_ids, mapping, usorted, pos, lane, tok);
    const uint32_t dests = __ballot_sync(0xffffffffu, myu >= 0);
    if (dests == 0) continue;
    const uint4* src = reinterpret_cast<const uint4*>(x + (tok >= 0 ? tok * H : 0));
    // every lane runs every batch (the shuffles below need the whole warp)
    for (int c0 = 0; c0 < pieces16; c0 += 32 * kBatch) {
      uint4 v[kBatch];
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        const int c = c0 + lane + 32 * j;
        v[j] = (tok >= 0 && c < pieces16 && c * 8 < H) ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
      }
      for (uint32_t m = dests; m; m &= m - 1) {
        const int64_t u = __shfl_sync(0xffffffffu, myu, __ffs(m) - 1);
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
          const int c = c0 + lane + 32 * j;
          if (c < pieces16) *reinterpret_cast<uint4*>(xs + ((int64_t)(c >> 3) * cap + u) * 64 + (c & 7) * 8) = v[j];
        }
      }
    }
  }
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < yacc_n4; i += (int64_t)gridDim.x * blockDim.x)
    reinterpret_cast<float4*>(yacc)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// Block-scaled FP8: gather_x_tok_kernel's work (x_sorted in bf16 for the LoRA
// shrink, y_acc zeroed) plus x quantised per row and 128-column group for the
// base GEMM: x8 [H/128][cap][128] E4M3 codes (zeros past H) and sx
// [H/128][cap] biased exponents (rows [n, cap): zero codes, exponent 127).
// Token-major (TOK: a token's groups are quantised once and written to the
// rows of its K pairs) or row-major, like gather_x_tok_kernel and
// gather_x_kernel.  Half a warp takes one group, eight values per lane.
template <bool TOK>
__global__ void __launch_bounds__(kGatherThreads)
gather_x_mx_kernel(const uint16_t* __restrict__ x, const int32_t* __restrict__ topk_ids,
                   const int32_t* __restrict__ mapping, const int32_t* __restrict__ usorted,
                   const int32_t* __restrict__ pos,
                   const uint32_t* __restrict__ n_valid, int T, int K, int E, int L, int H, int64_t cap,
                   uint16_t* __restrict__ xs, uint8_t* __restrict__ x8, uint8_t* __restrict__ sx,
                   float* __restrict__ yacc, int64_t yacc_n4) {
  pdl_wait();  // the predecessor on the stream has completed
  pdl_trigger();
  const int64_t n = *n_valid;
  const int64_t n_tasks = gather_tasks(T, K, n, cap, pos);
  const int lane = threadIdx.x & 31, half = lane >> 4, hl = lane & 15;
  const int64_t wpb = kGatherThreads / 32;
  const int ng = (H + 127) / 128;                 // groups per row
  const int pieces16 = (int)round_up(H, 64) / 8;  // 16-byte pieces of an x_sorted row
  const int64_t w0 = (int64_t)blockIdx.x * wpb + (threadIdx.x >> 5), ws = (int64_t)gridDim.x * wpb;
  constexpr int kPairs = 4;  // pairs of groups in flight per warp
  for (int64_t task = w0; task < n_tasks; task += ws) {
    int64_t tok;
    // TOK: lane j's destination row; else the one row is the task's
    const int myu = TOK ? gather_task_row(task, T, K, E, L, n, topk_ids, mapping, usorted, pos, lane, tok) : 0;
    if (!TOK) tok = task < n ? usorted[task] / K : -1;
    const uint32_t dests = TOK ? __ballot_sync(0xffffffffu, myu >= 0) : 1u;
    if (dests == 0) continue;
    const uint4* src = reinterpret_cast<const uint4*>(x + (tok >= 0 ? tok * H : 0));
    for (int g0 = 0; g0 < ng; g0 += 2 * kPairs) {
      uint4 v[kPairs];
#pragma unroll
      for (int j = 0; j < kPairs; ++j) {
        const int g = g0 + 2 * j + half, c = g * 16 + hl;  // c: 16-byte piece of the row
        v[j] = (tok >= 0 && g < ng && c * 8 < H) ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int j = 0; j < kPairs; ++j) {
        if (g0 + 2 * j >= ng) break;  // the same for both halves
        const int g = g0 + 2 * j + half, c = g * 16 + hl;
        const uint32_t wv[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
        uint32_t m = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) m = max(m, max(wv[k] & 0x7fffu, (wv[k] >> 16) & 0x7fffu));
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));  // within the half
        const int s = mx_group_exp_bf16(m);
        const float sc = exp2_neg(s);
        uint32_t q[2];
#pragma unroll
        for (int k = 0; k < 4; k += 2) {
          const uint32_t lo = f32x2_to_e4m3x2(__uint_as_float(wv[k] << 16) * sc, __uint_as_float(wv[k] & 0xffff0000u) * sc);
          const uint32_t hi =
              f32x2_to_e4m3x2(__uint_as_float(wv[k + 1] << 16) * sc, __uint_as_float(wv[k + 1] & 0xffff0000u) * sc);
          q[k / 2] = lo | (hi << 16);
        }
        for (uint32_t dm = dests; dm; dm &= dm - 1) {
          const int64_t u = TOK ? (int64_t)__shfl_sync(0xffffffffu, myu, __ffs(dm) - 1) : task;
          if (g < ng && c < pieces16)
            *reinterpret_cast<uint4*>(xs + ((int64_t)(c >> 3) * cap + u) * 64 + (c & 7) * 8) = v[j];
          if (g < ng) {
            *reinterpret_cast<uint2*>(x8 + ((int64_t)g * cap + u) * 128 + hl * 8) = make_uint2(q[0], q[1]);
            if (hl == 0) sx[(int64_t)g * cap + u] = (uint8_t)(s + 127);
          }
        }
      }
    }
  }
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < yacc_n4; i += (int64_t)gridDim.x * blockDim.x)
    reinterpret_cast<float4*>(yacc)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// acc[h][i] += A row h . member row i (h < NR, i < M) over k in [0, Kd): the
// warp streams NR rank rows at once, lanes strided in 16-byte pieces with
// NR x KB loads in flight; each A piece is unpacked once.  Rows may repeat.
template <int M, int NR, int KB>
__device__ __forceinline__ void gemv_dot(const uint16_t* const (&arow)[NR], const uint16_t* xr, int Kp, int Kd,
                                         int lane, float (&acc)[NR][kGemvRows]) {
  for (int k0 = lane * 8; k0 < Kd; k0 += 32 * 8 * KB) {
    uint4 av[NR][KB];
#pragma unroll
    for (int j = 0; j < KB; ++j) {
      const int k = k0 + j * 256;
#pragma unroll
      for (int h = 0; h < NR; ++h)
        av[h][j] = k < Kd ? __ldg(reinterpret_cast<const uint4*>(arow[h] + k)) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int j = 0; j < KB; ++j) {
      const int k = k0 + j * 256;
      if (k < Kd) {
        float af[NR][8];
#pragma unroll
        for (int h = 0; h < NR; ++h) {
          const uint32_t aw[4] = {av[h][j].x, av[h][j].y, av[h][j].z, av[h][j].w};
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            af[h][2 * w] = __uint_as_float(aw[w] << 16);
            af[h][2 * w + 1] = __uint_as_float(aw[w] & 0xffff0000u);
          }
        }
#pragma unroll
        for (int i = 0; i < M; ++i) {
          const uint4 xv = *reinterpret_cast<const uint4*>(xr + i * Kp + k);
          const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            const float x0 = __uint_as_float(xw[w] << 16), x1 = __uint_as_float(xw[w] & 0xffff0000u);
#pragma unroll
            for (int h = 0; h < NR; ++h) {
              acc[h][i] = fmaf(af[h][2 * w], x0, acc[h][i]);
              acc[h][i] = fmaf(af[h][2 * w + 1], x1, acc[h][i]);
            }
          }
        }
      }
    }
  }
}

// One warp's share of a bucket's rank rows, NR at a time: the dots with the m
// member rows, scaled by sc, into zv[(g * R16 + q) * kGemvRows + member].
template <int NG, int NR, int KB>
__device__ __forceinline__ void gemv_rows(const uint16_t* __restrict__ a, const uint16_t* xr, int Kp, int Kd, int l,
                                          int e, int E, int R, int R16, int r, int m, float sc, int warp, int lane,
                                          float* zv) {
  constexpr int kWarps = kGemvThreads / 32;
  const int nrows = NG * r;
  for (int task = NR * warp; task < nrows; task += NR * kWarps) {
    const uint16_t* arow[NR];
    int gq[NR];
#pragma unroll
    for (int h = 0; h < NR; ++h) {
      const int t = task + h < nrows ? task + h : task;  // past the end: repeat the first row
      const int g = t / r, q = t - g * r;
      gq[h] = g * R16 + q;
      arow[h] = a + ((((int64_t)l * E + e) * NG + g) * R + q) * (int64_t)Kd;
    }
    float acc[NR][kGemvRows];
#pragma unroll
    for (int h = 0; h < NR; ++h)
#pragma unroll
      for (int i = 0; i < kGemvRows; ++i) acc[h][i] = 0.f;
    static_assert(kGemvRows == 4, "one case per member count");
    switch (m) {  // uniform per CTA
      case 1: gemv_dot<1, NR, KB>(arow, xr, Kp, Kd, lane, acc); break;
      case 2: gemv_dot<2, NR, KB>(arow, xr, Kp, Kd, lane, acc); break;
      case 3: gemv_dot<3, NR, KB>(arow, xr, Kp, Kd, lane, acc); break;
      default: gemv_dot<4, NR, KB>(arow, xr, Kp, Kd, lane, acc); break;
    }
#pragma unroll
    for (int h = 0; h < NR; ++h) {
#pragma unroll
      for (int i = 0; i < kGemvRows; ++i)
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc[h][i] += __shfl_xor_sync(0xffffffffu, acc[h][i], o);
      if (lane < kGemvRows) {
        float v = acc[h][0];
#pragma unroll
        for (int i = 1; i < kGemvRows; ++i)
          if (lane == i) v = acc[h][i];
        zv[gq[h] * kGemvRows + lane] = sc * v;
      }
    }
  }
}

// CUDA-core shrink of buckets with at most kGemvRows pairs (NG rank blocks of
// LoRA A per adapter: 2 gate|up, 1 down).  One block per bucket (grid-stride
// over the listed buckets): the member rows are staged once in shared memory;
// each warp streams two (four, for short rows) rank rows of A at a time
// against them; then the block
// writes the bucket's whole z region with 16-byte stores (8 rank columns of
// one row each): s_l * dot for member rows and ranks q < r, zeros elsewhere.
// Dynamic shared memory: the member rows [kGemvRows][Kp] bf16, then the dots
// [NG * R16][kGemvRows] fp32.
template <int NG>
__global__ void __launch_bounds__(kGemvThreads)
shrink_gemv_kernel(const ShrinkRec* __restrict__ tiles, const int32_t* __restrict__ n_tiles,
                   const uint16_t* __restrict__ a, const uint16_t* __restrict__ rows, int Kd, int64_t cap,
                   int E, int R, int R16, const int32_t* __restrict__ lora_ranks,
                   const float* __restrict__ scalings, uint16_t* __restrict__ z, int64_t zcap) {
  pdl_wait();  // the predecessor on the stream has completed
  pdl_trigger();
  extern __shared__ __align__(16) uint8_t gemv_smem[];
  const int Kp = (Kd + 63) & ~63, kp8 = Kp / 8;
  uint16_t* xr = reinterpret_cast<uint16_t*>(gemv_smem);                      // [kGemvRows][Kp]
  float* zv = reinterpret_cast<float*>(gemv_smem + (size_t)kGemvRows * Kp * 2);  // [NG * R16][kGemvRows]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nt = *n_tiles;
  for (int tile = blockIdx.x; tile < nt; tile += gridDim.x) {
    const ShrinkRec t = tiles[tile];
    const int e = t.a.x, l = t.a.y, row0 = t.a.z, N = t.a.w;
    const int zrow0 = t.b.x, mlo = t.b.y, mhi = t.b.z;
    const int m = mhi - mlo;
    const int r = lora_ranks[l];
    const int r16 = (r + 15) & ~15;
    const float sc = scalings[l];
    __syncthreads();  // the previous bucket's reads of xr and zv are done
    for (int idx = threadIdx.x; idx < m * kp8; idx += kGemvThreads) {
      const int i = idx / kp8, c = idx - i * kp8;  // 16-byte piece c of member row i
      const int64_t u = (int64_t)row0 + mlo + i;
      *reinterpret_cast<uint4*>(xr + i * Kp + c * 8) =
          *reinterpret_cast<const uint4*>(rows + ((int64_t)(c >> 3) * cap + u) * 64 + (c & 7) * 8);
    }
    __syncthreads();
    // short rows (down shape, I <= 1024): four rank rows per warp at a time,
    // else two; either way about 6-8 KB of A in flight per warp
    if (Kd <= 1024) gemv_rows<NG, 4, 4>(a, xr, Kp, Kd, l, e, E, R, R16, r, m, sc, warp, lane, zv);
    else gemv_rows<NG, 2, 8>(a, xr, Kp, Kd, l, e, E, R, R16, r, m, sc, warp, lane, zv);
    __syncthreads();
    // the bucket's z region: N rows x (NG * r16 / 8) chunks of 8 rank columns
    const int cpg = r16 / 8, nchunk = NG * cpg;
    for (int idx = threadIdx.x; idx < N * nchunk; idx += kGemvThreads) {
      const int n = idx % N, c = idx / N, g = c / cpg, q8 = (c - g * cpg) * 8;
      const bool member = n >= mlo && n < mhi;
      uint32_t w[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int qa = q8 + 2 * j, qb = qa + 1;
        const float va = (member && qa < r) ? zv[(g * R16 + qa) * kGemvRows + (n - mlo)] : 0.f;
        const float vb = (member && qb < r) ? zv[(g * R16 + qb) * kGemvRows + (n - mlo)] : 0.f;
        w[j] = (uint32_t)f32_to_bf16_bits(va) | ((uint32_t)f32_to_bf16_bits(vb) << 16);
      }
      const int col0 = g * R16 + q8;  // a multiple of 8: one chunk of z
      *reinterpret_cast<uint4*>(z + ((int64_t)(col0 >> 3) * zcap + zrow0 + n) * 8) = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
}

// Deterministic top-k combine: y[t] = sum over k, in increasing k, of the
// pair rows dpair[t*K + k] (bf16 w * d written by the down GEMM), in fp32.
// Pairs the align dropped (expert or adapter id out of range) never received
// a row and add nothing.  One thread per 8 consecutive columns of a token; the
// rows of up to 8 pairs are loaded before any is added, so that a thread keeps
// 8 loads in flight (the sum still runs in increasing k).
__global__ void combine_kernel(const uint16_t* __restrict__ dpair, const int32_t* __restrict__ topk_ids,
                               const int32_t* __restrict__ mapping, int64_t T, int K, int H, int E, int L,
                               uint16_t* __restrict__ y) {
  pdl_wait();  // the predecessor on the stream has completed
  pdl_trigger();
  const int g8 = H / 8;
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= T * g8) return;
  const int64_t t = i / g8;
  const int c = (int)(i - t * g8) * 8;
  const int l = __ldg(mapping + t);
  const bool lora_ok = l >= -1 && l < L;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int k0 = 0; k0 < K; k0 += 8) {
    uint4 v[8];
    uint32_t ok = 0;  // bit j: pair k0 + j has a row
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int64_t pr = t * K + k0 + j;
      const int e = k0 + j < K ? __ldg(topk_ids + pr) : -1;
      const bool has = lora_ok && e >= 0 && e < E;
      ok |= has ? 1u << j : 0u;
      v[j] = has ? __ldg(reinterpret_cast<const uint4*>(dpair + pr * H + c)) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (!((ok >> j) & 1)) continue;
      const uint32_t wv[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        acc[2 * q] += __uint_as_float(wv[q] << 16);
        acc[2 * q + 1] += __uint_as_float(wv[q] & 0xffff0000u);
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

__global__ void convert_kernel(const float* __restrict__ yacc, uint16_t* __restrict__ y, int64_t n) {
  pdl_wait();  // the predecessor on the stream has completed
  pdl_trigger();
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

// LoRA A maps with 64/32/16/8-row boxes (m0, m2, m3, m4); a box taller than the
// tensor is skipped.  The 8-row map always exists (rows = L*E*R >= 8).
bool make_abox_maps(Maps& m, const void* base, uint64_t cols, uint64_t rows, int* mask) {
  CUtensorMap* slot[4] = {&m.m[kW], &m.m[kA32], &m.m[kA16], &m.m[kA8]};
  *mask = 0;
  for (int j = 0; j < 4; ++j) {
    const uint32_t bh = 64u >> j;
    if (bh > rows) continue;
    if (!make_map(slot[j], base, cols, rows, 64, bh, true)) return false;
    *mask |= 1 << j;
  }
  return (*mask & 8) != 0;
}

// 3-D bf16 view {d0, d1, d2} with byte strides s1 (dim 1) and s2 (dim 2).
bool make_map3(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t s1, uint64_t s2,
               uint32_t b0, uint32_t b1, uint32_t b2, bool swizzle128 = false) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {s1, s2};
  cuuint32_t box[3] = {b0, b1, b2};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 4-D bf16 view {d0..d3} with byte strides s1..s3, 128-byte swizzle.
bool make_map4(CUtensorMap* m, const void* base, const uint64_t (&d)[4], const uint64_t (&st)[3],
               const uint32_t (&b)[4], bool swizzle128 = true) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[4] = {d[0], d[1], d[2], d[3]};
  cuuint64_t strides[3] = {st[0], st[1], st[2]};
  cuuint32_t box[4] = {b[0], b[1], b[2], b[3]};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Row-operand maps with 128-, 256- and 192-row boxes over a chunk-major buffer
// of `rows` 64-column rows; returns the mask of the maps made (a box taller
// than the buffer is skipped).
bool make_row_maps(Maps& m, const void* base, uint64_t rows, int* mask) {
  *mask = 0;
  const int slot[3] = {kRows128, kRows256, kRows192};
  const uint32_t height[3] = {128, 256, 192};
  for (int j = 0; j < 3; ++j) {
    if (rows < height[j]) continue;
    if (!make_map(&m.m[slot[j]], base, 64, rows, 64, height[j], true)) return false;
    *mask |= 1 << j;
  }
  return true;
}

// Half-tile row maps of the pair kinds: 32-, 96- and 128-row boxes (the
// 64-row box is kRows) over a chunk-major buffer of `rows` >= 128 rows.
bool make_pair_row_maps(Maps& m, const void* base, uint64_t rows) {
  const int slot[3] = {kRh32, kRh96, kRows128};
  const uint32_t height[3] = {32, 96, 128};
  for (int j = 0; j < 3; ++j)
    if (rows < height[j] || !make_map(&m.m[slot[j]], base, 64, rows, 64, height[j], true)) return false;
  return true;
}

// Maps of the gate_up-shape shrink (two rank blocks per adapter): the row
// operand `rows` (chunk-major [ceil(Kd/64)][cap][64]) and LoRA A as
// [L, E, 2, R, Kd].  Returns the masks of the optional views it made.
bool make_shrink2_maps(Maps& m, const void* rows, uint64_t cap, int Kd, const void* lora_a, int L, int E, int R,
                       int* abox, int* a3, int* aw, int* rmask) {
  const uint64_t kc = (uint64_t)ceil_div(Kd, 64);
  *abox = *a3 = *aw = *rmask = 0;
  bool ok = make_map(&m.m[kRows], rows, 64, kc * cap, 64, 64, true) && make_row_maps(m, rows, kc * cap, rmask) &&
            // x rows as [chunk][row][64]: a box of 64 or 128 rows covers two K chunks
            make_map3(&m.m[kX2x64], rows, 64, cap, kc, 128, cap * 128, 64, 64, 2, true) &&
            make_map3(&m.m[kX2x128], rows, 64, cap, kc, 128, cap * 128, 64, 128, 2, true);
  *rmask &= 1;  // shrink tiles hold at most 128 rows
  if (!ok || L == 0) return ok;
  for (int j = 0; ok && j < 3; ++j) {
    const uint32_t rb = 16u << j;
    if ((int)rb > R) continue;
    // wide boxes: rb gate and rb up rank rows of two K chunks; exact only when
    // Kd is a multiple of 64 (else the last chunk of the last row would run past
    // the tensor)
    if (Kd % 64 == 0) {
      const uint64_t d[4] = {64, (uint64_t)R, (uint64_t)L * E * 2, (uint64_t)Kd / 64};
      const uint64_t st[3] = {(uint64_t)Kd * 2, (uint64_t)R * Kd * 2, 128};
      const uint32_t b[4] = {64, rb, 2, 2};
      ok = make_map4(&m.m[kAW16 + j], lora_a, d, st, b);
      *aw |= 1 << j;
    }
    // LoRA A as [(l, e, gate|up)][rank][k]: a box {64, rb, 2} holds rb gate and rb up rank rows
    ok = ok && make_map3(&m.m[kA3x16 + j], lora_a, Kd, R, (uint64_t)L * E * 2, (uint64_t)Kd * 2,
                         (uint64_t)R * Kd * 2, 64, rb, 2, true);
    *a3 |= 1 << j;
  }
  return ok && make_abox_maps(m, lora_a, Kd, (uint64_t)L * E * 2 * R, abox);
}

// Maps of the down-shape shrink (one rank block per adapter): the row operand
// and LoRA A as [L, E, R, Kd].
bool make_shrink1_maps(Maps& m, const void* rows, uint64_t cap, int Kd, const void* lora_a, int L, int E, int R,
                       int* abox, int* aw, int* rmask) {
  const uint64_t kc = (uint64_t)ceil_div(Kd, 64);
  *abox = *aw = *rmask = 0;
  bool ok = make_map(&m.m[kRows], rows, 64, kc * cap, 64, 64, true) && make_row_maps(m, rows, kc * cap, rmask) &&
            make_map3(&m.m[kX2x64], rows, 64, cap, kc, 128, cap * 128, 64, 64, 2, true) &&
            make_map3(&m.m[kX2x128], rows, 64, cap, kc, 128, cap * 128, 64, 128, 2, true);
  *rmask &= 1;
  if (!ok || L == 0) return ok;
  for (int j = 0; ok && j < 3; ++j) {
    const uint32_t rb = 16u << j;
    if ((int)rb > R || Kd % 64 != 0) continue;
    ok = make_map3(&m.m[kAW16 + j], lora_a, 64, (uint64_t)L * E * R, (uint64_t)Kd / 64, (uint64_t)Kd * 2, 128, 64,
                   rb, 2, true);
    *aw |= 1 << j;
  }
  return ok && make_abox_maps(m, lora_a, Kd, (uint64_t)L * E * R, abox);
}

// Maps of the down-shape GEMM on CTA pairs: weights as [E * M rows][Kd], the
// row operand (chunk-major, half-tile boxes of 32 / 64 / 96 / 128 rows), LoRA
// B as [L, E, M, R] in rank chunks of 8, and z (chunk-major
// [zchunks][zcap][8]) in half-piece boxes.
bool make_down_maps(Maps& m, const void* w, int M, int Kd, int E, const void* rows, uint64_t cap,
                    const void* lora_b, int L, int R, const void* z, uint64_t zcap, int zchunks) {
  const uint64_t kc = (uint64_t)ceil_div(Kd, 64);
  bool ok = make_map(&m.m[kW], w, Kd, (uint64_t)E * M, 64, 128, true) &&
            make_map(&m.m[kRows], rows, 64, kc * cap, 64, 64, true) && make_pair_row_maps(m, rows, kc * cap);
  if (!ok || L == 0) return ok;
  const int nc[3] = {8, 4, 2};
  const int bslot[3] = {kB8, kB4, kB2}, zslot[3] = {kZ8, kZ4, kZ2}, zsslot[3] = {kZ8s, kZ4s, kZ2s};
  for (int j = 0; ok && j < 3; ++j) {
    if (nc[j] > R / 8) continue;  // a box may not span more rank chunks than exist
    ok = make_map3(&m.m[bslot[j]], lora_b, 8, (uint64_t)L * E * M, (uint64_t)R / 8, (uint64_t)R * 2, 16, 8, 128,
                   nc[j]) &&
         make_map3(&m.m[zslot[j]], z, 8, zcap, (uint64_t)zchunks, 16, zcap * 16, 8, 128, nc[j]) &&
         make_map3(&m.m[zsslot[j]], z, 8, zcap, (uint64_t)zchunks, 16, zcap * 16, 8, 64, nc[j]);
  }
  return ok;
}

// Bit 0 / 1: the 8- / 4-chunk LoRA B and z views exist (they need R / 8 chunks).
int b_view_mask(int R) { return (R / 8 >= 8 ? 1 : 0) | (R / 8 >= 4 ? 2 : 0); }

constexpr int kMaxForwardBuckets = 16384;  // E * (L + 1): the plan keeps two scans of it in shared memory

struct FwdLayout {
  bool ok;
  AlignPlan al;
  int R16, C, mtiles_gu, mtiles_d;
  int64_t cap, zcap, max_base, max_shrink, max_pieces, max_gemv;
  int64_t o_align, o_base, o_shrink, o_gemv, o_pieces, o_ustart, o_usorted, o_pos,
      o_counts, o_zgu, o_h, o_zd, o_yacc, o_xs, o_x8, o_sx, o_h8, o_sh, total;
};

// act_q (block-scaled FP8): also the quantised x and h with their exponents.
FwdLayout fwd_layout(int32_t T, int32_t K, int32_t E, int32_t H, int32_t I, int32_t L, int32_t R,
                     bool act_q = false) {
  FwdLayout f{};
  f.ok = false;
  if (T < 0 || K < 1 || E < 1 || H < 128 || I < 64 || L < 0 || R < 0) return f;
  if (H % 8 || I % 8 || R > 256 || (L > 0 && (R % 16 != 0 || R < 16))) return f;
  f.al = align_plan(T, K, E, L, kBlock);
  if (!f.al.ok || f.al.NB > kMaxForwardBuckets) return f;
  f.R16 = (int)round_up(R, 16);
  if (f.R16 == 0) f.R16 = 16;
  f.C = L + 1;
  f.mtiles_gu = (int)ceil_div(2 * f.R16, 128);
  f.mtiles_d = (int)ceil_div(f.R16, 128);
  const int64_t P = f.al.P;
  const int64_t nb_nonempty = P < f.al.NB ? P : f.al.NB;
  // dense rows plus room for a 256-row box from the last 16-aligned tile start
  f.cap = round_up(P, 16) + kTileRows;
  // z regions: each non-empty LoRA bucket adds < 32 rows of 16-row alignment
  f.zcap = round_up(P + 32 * nb_nonempty, 16) + kTileRows;
  f.max_base = P / kMxTileRows + 2 * (int64_t)E + 1;  // tiles of at most 256 (or kMxTileRows) rows
  f.max_shrink = (P + 32 * nb_nonempty) / kShrinkRows + nb_nonempty + 1;
  f.max_pieces = nb_nonempty + f.max_base;
  f.max_gemv = nb_nonempty;
  if (f.cap * round_up(H > I ? H : I, 64) >= ((int64_t)1 << 31) || f.zcap * 2 * f.R16 >= ((int64_t)1 << 31)) return f;
  int64_t o = 0;
  auto take = [&](int64_t bytes) { const int64_t r = o; o += round_up(bytes > 0 ? bytes : 1, 256); return r; };
  f.o_align = take(f.al.ws_bytes);
  f.o_base = take(f.max_base * (int64_t)sizeof(TileRec));
  f.o_shrink = take(f.max_shrink * (int64_t)sizeof(ShrinkRec));
  f.o_gemv = take(f.max_gemv * (int64_t)sizeof(ShrinkRec));
  f.o_pieces = take(f.max_pieces * 16);
  f.o_ustart = take(((int64_t)f.al.NB + 1) * 4);
  f.o_usorted = take(f.cap * 4);
  f.o_pos = take(P * 4);  // dense row of each pair, for the token-major gathers
  f.o_counts = take(16);
  f.o_zgu = take(f.zcap * 2 * f.R16 * 2);
  f.o_h = take(f.cap * round_up(I, 64) * 2);
  f.o_zd = take(f.zcap * f.R16 * 2);
  f.o_yacc = take((int64_t)T * H * 4);
  f.o_xs = take(f.cap * round_up(H, 64) * 2);
  if (act_q) {
    f.o_x8 = take(f.cap * round_up(H, 128));
    f.o_sx = take(ceil_div(H, 128) * f.cap);
    f.o_h8 = take(f.cap * round_up(I, 128));
    f.o_sh = take(ceil_div(I, 128) * f.cap);
  }
  f.total = o;
  f.ok = true;
  return f;
}

// The current device, or -1 when it cannot be read or is beyond the 64
// devices the per-device caches below hold.
int current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -1;
  return dev;
}

int sm_count() {
  static int n[64] = {};
  const int dev = current_device();
  if (dev < 0) return 148;
  if (n[dev] == 0) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = 148;
    n[dev] = v;
  }
  return n[dev];
}

// Persistent launch: one CTA per SM, or for the pair kinds as many clusters of
// two as are resident at once (fewer when there are fewer items).
template <int KIND, int QF = kQNone>
int launch_gemm(const Maps& maps, const Params& p, int64_t max_tiles, cudaStream_t stream) {
  static_assert(smem_bytes<KIND, QF>() <= 227 * 1024, "shared memory per CTA");
  const int smem = smem_bytes<KIND, QF>();
  // the shared-memory opt-in and the resident-cluster count are per device
  const int dev = current_device();
  static bool configured[64] = {};
  if (dev < 0 || !configured[dev]) {
    if (cudaFuncSetAttribute(moe_gemm_kernel<KIND, QF>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
        cudaSuccess)
      return MLR_ERR_CUDA;
    if (dev >= 0) configured[dev] = true;
  }
  const int64_t max_items = max_tiles * p.nblk;
  if (max_items <= 0) return MLR_OK;
  if (max_items > INT32_MAX) return MLR_ERR_UNSUPPORTED;
  if (kPairOf<KIND, QF>) {
    // clusters of two CTAs, as many as can be resident at once (a persistent
    // grid with one pair more than fits would run that pair after the others)
    // (and programmatic stream serialization, see pdl_wait)
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kLaunchThreads<KIND, QF>);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;  // the occupancy query below takes the cluster shape only
    static int resident_of[64] = {};
    int resident = dev >= 0 ? resident_of[dev] : 0;
    if (resident == 0) {
      cfg.gridDim = dim3(2 * (unsigned)(sm_count() / 2));
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, moe_gemm_kernel<KIND, QF>, &cfg) != cudaSuccess || n <= 0)
        return MLR_ERR_CUDA;
      resident = n;
      if (dev >= 0) resident_of[dev] = n;
    }
    const int64_t pairs = max_items < resident ? max_items : resident;
    cfg.gridDim = dim3(2 * (unsigned)pairs);
    cfg.numAttrs = 2;
    if (cudaLaunchKernelEx(&cfg, moe_gemm_kernel<KIND, QF>, maps, p) != cudaSuccess) return MLR_ERR_CUDA;
  } else {
    const int grid = (int)(max_items < sm_count() ? max_items : sm_count());
    if (launch_pdl(moe_gemm_kernel<KIND, QF>, dim3(grid), dim3(kLaunchThreads<KIND, QF>), smem, stream, maps, p) != cudaSuccess) return MLR_ERR_CUDA;
    MLR_CHECK_LAUNCH();
  }
  note_launch();
  return MLR_OK;
}

// CUDA-core shrink of the small buckets: each CTA takes listed buckets in a
// grid-stride loop up to the device-side count.
template <int NG>
int launch_gemv(const ShrinkRec* tiles, const int32_t* n_tiles, int64_t max_tiles, const void* a, const uint16_t* rows,
                int Kd, const FwdLayout& f, int E, int R, const int32_t* lora_ranks, const float* scalings,
                uint16_t* z, cudaStream_t stream) {
  if (max_tiles <= 0) return MLR_OK;
  const int smem = kGemvRows * (int)round_up(Kd, 64) * 2 + NG * f.R16 * kGemvRows * 4;
  const int dev = current_device();
  static int configured[64] = {};  // largest opt-in so far, per device
  if (smem > 48 * 1024 && (dev < 0 || smem > configured[dev])) {
    if (cudaFuncSetAttribute(shrink_gemv_kernel<NG>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
        cudaSuccess)
      return MLR_ERR_CUDA;
    if (dev >= 0) configured[dev] = smem;
  }
  const int64_t grid = max_tiles < 8 * (int64_t)sm_count() ? max_tiles : 8 * (int64_t)sm_count();
  if (launch_pdl(shrink_gemv_kernel<NG>, dim3((unsigned)grid), dim3(kGemvThreads), smem, stream, 
      tiles, n_tiles, static_cast<const uint16_t*>(a), rows, Kd, f.cap, E, R, f.R16, lora_ranks, scalings, z,
      f.zcap) != cudaSuccess) return MLR_ERR_CUDA;
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

extern "C" size_t fused_moe_lora_workspace_bytes_fp8_w8a8(int32_t num_tokens, int32_t topk, int32_t num_experts,
                                                         int32_t hidden, int32_t intermediate, int32_t num_loras,
                                                         int32_t max_rank) {
  const mlr::FwdLayout f =
      mlr::fwd_layout(num_tokens, topk, num_experts, hidden, intermediate, num_loras, max_rank, true);
  return f.ok ? (size_t)f.total : 0;
}

namespace mlr {
namespace {

// 3-D uint8 view {d0, d1, d2} with byte strides s1 (dim 1) and s2 (dim 2), no
// swizzle (FP8 weight codes, read by the converters as plain rows).
bool make_map3_u8(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t s1,
                  uint64_t s2, uint32_t b0, uint32_t b1, uint32_t b2) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {s1, s2};
  cuuint32_t box[3] = {b0, b1, b2};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The layer.  qf = kQFp8 / kQInt8: w_gate_up / w_down hold E4M3 / INT8 codes
// with block scales s_gu [E][ceil(2I/128)][ceil(H/128)] and s_d
// [E][ceil(H/128)][ceil(I/128)]; kQU4: two UINT4 codes per byte ([E][2I][H/2]
// and [E][H][I/2]) with group scales and zero points s_gu, z_gu
// [E][2I][ceil(H/128)] and s_d, z_d [E][H][ceil(I/128)]; kQMx: E4M3 codes
// with power-of-two block scales given as biased exponents in z_gu
// [E][ceil(2I/128)][ceil(H/128)] and z_d [E][ceil(H/128)][ceil(I/128)], the
// activations quantised on the way (s_gu, s_d unused); kQNone: bf16, the
// scales unused.
int moe_forward(const mlr_bf16* x, const int32_t* topk_ids, const float* topk_weights,
                const int32_t* token_lora_mapping, const int32_t* lora_ranks, const float* scalings,
                const void* w_gate_up, const void* w_down, const float* s_gu, const float* s_d,
                const uint8_t* z_gu, const uint8_t* z_d, int qf,
                const mlr_bf16* lora_a_gu, const mlr_bf16* lora_b_gu, const mlr_bf16* lora_a_down,
                const mlr_bf16* lora_b_down, int32_t T, int32_t K, int32_t E, int32_t H, int32_t I, int32_t L,
                int32_t R, mlr_bf16* y, void* workspace, size_t ws_bytes, int32_t* d_status,
                cudaStream_t stream) {
  const bool mx = qf == kQMx;
  const FwdLayout f = fwd_layout(T, K, E, H, I, L, R, mx);
  if (!f.ok) {
    if (T < 0 || K < 1 || E < 1 || L < 0 || R < 0) return MLR_ERR_INVALID;
    return MLR_ERR_UNSUPPORTED;
  }
  const bool quant = qf != kQNone;
  // Codes are one byte (half a byte for UINT4): the TMA row strides (H and I
  // codes) must be 16-byte multiples
  const int cmul = qf == kQU4 ? 32 : 16;
  if (quant && (H % cmul != 0 || I % cmul != 0)) return MLR_ERR_UNSUPPORTED;
  if (T == 0) return MLR_OK;
  const void* need[] = {x, topk_ids, topk_weights, token_lora_mapping, w_gate_up, w_down, y};
  for (const void* q : need)
    if (q == nullptr) return MLR_ERR_INVALID;
  if (quant && !mx && (s_gu == nullptr || s_d == nullptr || (reinterpret_cast<uintptr_t>(s_gu) & 3) != 0 ||
                (reinterpret_cast<uintptr_t>(s_d) & 3) != 0))
    return MLR_ERR_INVALID;
  if ((qf == kQU4 || mx) && (z_gu == nullptr || z_d == nullptr)) return MLR_ERR_INVALID;
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
  char* aws = ws + f.o_align;
  TileRec* base_tiles = reinterpret_cast<TileRec*>(ws + f.o_base);
  ShrinkRec* shrink_tiles = reinterpret_cast<ShrinkRec*>(ws + f.o_shrink);
  ShrinkRec* gemv_tiles = reinterpret_cast<ShrinkRec*>(ws + f.o_gemv);
  int4* pieces = reinterpret_cast<int4*>(ws + f.o_pieces);
  uint32_t* ustart = reinterpret_cast<uint32_t*>(ws + f.o_ustart);
  int32_t* usorted = reinterpret_cast<int32_t*>(ws + f.o_usorted);
  int32_t* counts = reinterpret_cast<int32_t*>(ws + f.o_counts);
  uint16_t* zgu = reinterpret_cast<uint16_t*>(ws + f.o_zgu);
  uint16_t* hbuf = reinterpret_cast<uint16_t*>(ws + f.o_h);
  uint16_t* zd = reinterpret_cast<uint16_t*>(ws + f.o_zd);
  float* yacc = reinterpret_cast<float*>(ws + f.o_yacc);
  uint16_t* xs = reinterpret_cast<uint16_t*>(ws + f.o_xs);
  uint8_t* x8 = mx ? reinterpret_cast<uint8_t*>(ws + f.o_x8) : nullptr;
  uint8_t* sx = mx ? reinterpret_cast<uint8_t*>(ws + f.o_sx) : nullptr;
  uint8_t* h8 = mx ? reinterpret_cast<uint8_t*>(ws + f.o_h8) : nullptr;
  uint8_t* sh = mx ? reinterpret_cast<uint8_t*>(ws + f.o_sh) : nullptr;
  const uint32_t* btotal = reinterpret_cast<const uint32_t*>(aws + f.al.btotal_off);

  // tensor maps
  Maps m_sgu{}, m_gu{}, m_sd{}, m_dn{};
  int abox_gu = 0, abox_d = 0, a3_gu = 0, w3 = 0, aw_gu = 0, aw_d = 0;
  int rm_sgu = 0, rm_gu = 0, rm_sd = 0, rm_dn = 0;
  const int bmask = L > 0 ? b_view_mask(R) : 0;
  const uint64_t cap = (uint64_t)f.cap, zcap = (uint64_t)f.zcap;
  const uint64_t hk = (uint64_t)ceil_div(H, 64);
  const uint32_t zrows = (uint32_t)(f.zcap < 256 ? f.zcap : 256);
  bool ok = make_map(&m_gu.m[kW], w_gate_up, H, (uint64_t)E * 2 * I, 64, 128, true) &&
            make_map(&m_gu.m[kRows], xs, 64, hk * cap, 64, 64, true) &&
            // bf16 gate_up runs on CTA pairs (half-tile row boxes); the others take whole tiles
            (qf == kQNone ? make_pair_row_maps(m_gu, xs, hk * cap) : make_row_maps(m_gu, xs, hk * cap, &rm_gu)) &&
            make_shrink2_maps(m_sgu, xs, cap, H, lora_a_gu, L, E, R, &abox_gu, &a3_gu, &aw_gu, &rm_sgu) &&
            make_shrink1_maps(m_sd, hbuf, cap, I, lora_a_down, L, E, R, &abox_d, &aw_d, &rm_sd) &&
            make_down_maps(m_dn, w_down, H, I, E, hbuf, cap, lora_b_down, L, R, zd, zcap, f.R16 / 8);
  if (ok && I >= 128 && !quant) {
    // W_gate_up as [(e, gate|up)][row][k]: a box {64, 128, 2} is a 128-row block of gate and of up
    ok = make_map3(&m_gu.m[kW3], w_gate_up, H, I, (uint64_t)E * 2, (uint64_t)H * 2, (uint64_t)I * H * 2, 64, 128, 2,
                   true);
    w3 = 1;
  }
  if (ok && mx) {
    // E4M3 codes mapped as 2-byte elements: 128 bytes = 64 elements per K step
    // with the bf16 kernels' 128-byte swizzle.  W_gate_up as [(e, gate|up)][I
    // rows][H/2] (a box is a 128-row block of gate and of up), W_down as [E*H
    // rows][I/2], the quantised x and h as [K/128 chunk][cap rows][64]; the
    // single-CTA down GEMM takes whole-tile row boxes over h.  Codes past H
    // (or I) and rows past I (or H) read 0.
    const uint64_t hk8 = (uint64_t)ceil_div(H, 128), ik8 = (uint64_t)ceil_div(I, 128);
    ok = make_map3(&m_gu.m[kW3], w_gate_up, (uint64_t)H / 2, I, (uint64_t)E * 2, (uint64_t)H, (uint64_t)I * H, 64,
                   128, 2, true) &&
         make_map(&m_gu.m[kRows], x8, 64, hk8 * cap, 64, 64, true) && make_row_maps(m_gu, x8, hk8 * cap, &rm_gu) &&
         make_map(&m_dn.m[kW], w_down, (uint64_t)I / 2, (uint64_t)E * H, 64, 256, true) &&
         make_map(&m_dn.m[kRows], h8, 64, ik8 * cap, 64, 64, true) && make_row_maps(m_dn, h8, ik8 * cap, &rm_dn);
    w3 = 1;
  } else if (ok && quant) {
    // codes: W_gate_up as [(e, gate|up)][I rows][row bytes], a box of one K step's bytes (64, or 32
    // for UINT4) x 128 rows of gate and of up; W_down as [e][H rows][row bytes], a box of one K
    // step's bytes x 128 rows.  Rows past I (or H) read 0.
    const uint64_t hb = qf == kQU4 ? (uint64_t)H / 2 : (uint64_t)H, ib = qf == kQU4 ? (uint64_t)I / 2 : (uint64_t)I;
    const uint32_t kbox = qf == kQU4 ? 32 : 64;
    ok = make_map3_u8(&m_gu.m[kW], w_gate_up, hb, I, (uint64_t)E * 2, hb, (uint64_t)I * hb, kbox, 128, 2) &&
         make_map3_u8(&m_dn.m[kW], w_down, ib, H, E, ib, (uint64_t)H * ib, kbox, 128, 1) &&
         // the FP8 down GEMM runs on single CTAs: whole-tile row boxes over h, and
         // z boxes of zrows rows (a CTA loads a piece's z rows whole)
         make_row_maps(m_dn, hbuf, (uint64_t)ceil_div(I, 64) * cap, &rm_dn);
  }
  if (ok && quant) {
    const int nc[3] = {8, 4, 2};
    const int zslot[3] = {kZ8, kZ4, kZ2};
    for (int j = 0; ok && L > 0 && j < 3; ++j) {
      if (nc[j] > R / 8) continue;
      ok = make_map3(&m_dn.m[zslot[j]], zd, 8, zcap, (uint64_t)f.R16 / 8, 16, zcap * 16, 8, zrows, nc[j]);
    }
  }
  // z rows per box of the gate_up expand: a CTA of a pair loads half of a
  // piece's rows (at most 128), a single CTA all of them
  const uint32_t zr_gu = qf == kQNone ? 128u : zrows;
  if (ok && L > 0) {
    // gate_up expand: LoRA B stacks as [rank chunk][row][8] (each row's ranks are
    // contiguous) and chunk-major z [column/8][zcap][8]
    const int nc[3] = {8, 4, 2};
    const int bslot[3] = {kB8, kB4, kB2}, zslot[3] = {kZ8, kZ4, kZ2}, zsslot[3] = {kZ8s, kZ4s, kZ2s};
    for (int j = 0; ok && j < 3; ++j) {
      if (nc[j] > R / 8) continue;  // a box may not span more rank chunks than exist
      ok = make_map3(&m_gu.m[bslot[j]], lora_b_gu, 8, (uint64_t)L * E * 2 * I, (uint64_t)R / 8, (uint64_t)R * 2, 16,
                     8, 128, nc[j]) &&
           make_map3(&m_gu.m[zslot[j]], zgu, 8, zcap, (uint64_t)2 * f.R16 / 8, 16, zcap * 16, 8, zr_gu, nc[j]) &&
           make_map3(&m_gu.m[zsslot[j]], zgu, 8, zcap, (uint64_t)2 * f.R16 / 8, 16, zcap * 16, 8, 64, nc[j]);
    }
  }
  // joint gate+up expand steps: LoRA B as [(l, e, gate|up)][chunk][I rows][8]
  // (a box holds 128 rows of a gate and of an up block: I >= 128) and z as
  // [gate|up][chunk][zcap][8] (its two column halves)
  int gu_joint = 0;
  if (ok && L > 0 && I >= 128 && zrows >= 64) {
    const uint32_t nc[3] = {8, 4, 2};
    const int bslot[3] = {kBJ8, kBJ4, kBJ2}, zslot[3] = {-1, kZJ4, kZJ2}, zsslot[3] = {kZJ8s, kZJ4s, kZJ2s};
    const uint64_t rc16 = (uint64_t)f.R16 / 8;
    for (int j = 0; ok && j < 3; ++j) {
      if (nc[j] > (uint32_t)(R / 8)) continue;
      const uint64_t bd[4] = {8, (uint64_t)I, (uint64_t)R / 8, (uint64_t)L * E * 2};
      const uint64_t bst[3] = {(uint64_t)R * 2, 16, (uint64_t)I * R * 2};
      const uint64_t zd4[4] = {8, zcap, rc16, 2};
      const uint64_t zst[3] = {16, zcap * 16, rc16 * zcap * 16};
      ok = make_map4(&m_gu.m[bslot[j]], lora_b_gu, bd, bst, {8, 128, nc[j], 2}, false) &&
           make_map4(&m_gu.m[zsslot[j]], zgu, zd4, zst, {8, 64, nc[j], 2}, false) &&
           (zslot[j] < 0 || make_map4(&m_gu.m[zslot[j]], zgu, zd4, zst, {8, zr_gu, nc[j], 2}, false));
    }
    gu_joint = ok ? 1 : 0;
  }
  if (!ok) return MLR_ERR_CUDA;

  // deterministic combine: the down GEMM writes each pair's weighted row into
  // the x_sorted region (dead after gate_up: P rows of H <= its cap rows of
  // round_up(H, 64)) and a combine kernel sums a token's rows in k order
  const bool det = combine_deterministic();
  const int prof = prof_call_begin(stream);
  int rc = MLR_OK;
  // the CUDA-core shrink pays off when buckets average a few pairs (decode)
  const int64_t nb_nonempty = f.al.P < f.al.NB ? f.al.P : f.al.NB;
  const int gemv_rows = (L > 0 && f.al.P < 8 * nb_nonempty) ? kGemvRows : 0;
  // largest experts first when experts average more than 32 rows (several
  // tiles of differing sizes); small batches keep the cheaper plain order
  const int by_span = f.al.P > 32 * (int64_t)E ? 1 : 0;
  const int max_rows = mx ? kMxTileRows : kTileRows;  // rows per base tile
  const size_t scan_bytes = (size_t)round_up(((int64_t)f.al.NB + 1) * 4, 16);
  if (align_block_ok(f.al, scan_bytes)) {
    // one launch: the dense align and the tile plan (timed as the align stage)
    const size_t zs_off = align_block_smem(f.al), sm = zs_off + scan_bytes;
    if (sm > 48 * 1024 &&
        cudaFuncSetAttribute(align_plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)sm) != cudaSuccess)
      return MLR_ERR_CUDA;
    if (launch_pdl(align_plan_kernel, dim3(1), dim3(kPlanThreads), sm, stream, topk_ids, token_lora_mapping, (int)f.al.P, K, E, L, R,
                                                       lora_ranks, usorted, ustart, base_tiles, pieces,
                                                       shrink_tiles, gemv_tiles, counts, d_status, (int)zs_off,
                                                       gemv_rows, by_span, max_rows, gu_joint) != cudaSuccess) return MLR_ERR_CUDA;
    MLR_CHECK_LAUNCH();
    note_launch();
    prof_mark(prof, 0, stream);
  } else {
    // chunked: per-chunk counts, the plan (which scans the bucket sizes into
    // the dense starts), then the dense scatter
    if ((rc = align_dense_count(f.al, topk_ids, token_lora_mapping, K, E, L, aws, d_status, stream)) != MLR_OK)
      return rc;
    const size_t sm = 2 * scan_bytes;
    if (sm > 48 * 1024 &&
        cudaFuncSetAttribute(plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm) != cudaSuccess)
      return MLR_ERR_CUDA;
    if (launch_pdl(plan_kernel, dim3(1), dim3(kPlanThreads), sm, stream, btotal, lora_ranks, E, f.C, R, ustart, base_tiles, pieces,
                                                  shrink_tiles, gemv_tiles, counts, d_status, gemv_rows,
                                                  by_span, max_rows, gu_joint) != cudaSuccess) return MLR_ERR_CUDA;
    MLR_CHECK_LAUNCH();
    note_launch();
    if ((rc = align_dense_scatter(f.al, topk_ids, token_lora_mapping, K, E, L, aws, ustart, usorted, stream)) !=
        MLR_OK)
      return rc;
    prof_mark(prof, 0, stream);
  }
  {
    // Row by row of x_sorted, each reading its token's row of x: the K rows
    // of a token read it at scattered times, from L2 while x_sorted's writes
    // leave it there.  Where they stream more than twice the 129 MB L2, the
    // dense row of each pair is found first and x_sorted is written token by
    // token (each row of x read once for its K pairs).
    const bool tok_major = (int64_t)f.al.P * round_up(H, 64) * 2 > ((int64_t)256 << 20);
    int32_t* pos = tok_major ? reinterpret_cast<int32_t*>(ws + f.o_pos) : nullptr;
    if (tok_major) {
      const int64_t pblocks = ceil_div(f.al.P, kGatherThreads);
      if (launch_pdl(dense_pos_kernel, dim3((unsigned)(pblocks < 4 * sm_count() ? pblocks : 4 * sm_count())),
                     dim3(kGatherThreads), 0, stream, usorted, ustart + f.al.NB, pos) != cudaSuccess)
        return MLR_ERR_CUDA;
      MLR_CHECK_LAUNCH();
      note_launch();
    }
    // (the kernels stride over their tasks; the padding rows number cap - n >= cap - P)
    const int64_t tasks = tok_major ? (int64_t)T * ceil_div(K, 32) + (f.cap - f.al.P) : f.cap;
    const int64_t blocks = ceil_div(tasks > 0 ? tasks : 1, kGatherThreads / 32);
    const int grid = (int)(blocks < 16 * sm_count() ? blocks : 16 * sm_count());
    const cudaError_t e =
        mx ? launch_pdl(tok_major ? gather_x_mx_kernel<true> : gather_x_mx_kernel<false>, dim3(grid),
                        dim3(kGatherThreads), 0, stream, x, topk_ids, token_lora_mapping, (const int32_t*)usorted,
                        (const int32_t*)pos, ustart + f.al.NB, T, K, E, L, H, f.cap, xs, x8, sx, yacc,
                        det ? 0 : (int64_t)T * H / 4)
           : tok_major
               ? launch_pdl(gather_x_tok_kernel, dim3(grid), dim3(kGatherThreads), 0, stream, x, topk_ids,
                            token_lora_mapping, (const int32_t*)usorted, (const int32_t*)pos, ustart + f.al.NB, T, K,
                            E, L, H, f.cap, xs, yacc, det ? 0 : (int64_t)T * H / 4)
               : launch_pdl(gather_x_kernel, dim3(grid), dim3(kGatherThreads), 0, stream, x, usorted,
                            ustart + f.al.NB, K, H, f.cap, xs, yacc, det ? 0 : (int64_t)T * H / 4);
    if (e != cudaSuccess) return MLR_ERR_CUDA;
    MLR_CHECK_LAUNCH();
    note_launch();
  }
  prof_mark(prof, 1, stream);

  Params p{};
  p.T = T; p.K = K; p.E = E; p.H = H; p.I = I; p.L = L; p.R = R; p.R16 = f.R16; p.C = f.C;
  p.cap = (int)f.cap;
  p.zcap = (int)f.zcap;
  p.zrows = (int)zrows;
  p.zshort = zrows >= 64 ? 1 : 0;  // zcap >= 256, so the 64-row maps always exist
  p.bmask = bmask;
  p.gu_joint = gu_joint;
  p.P = (int64_t)T * K;
  p.wait_ns = wait_limit_ns();
  p.topk_weights = topk_weights;
  p.lora_ranks = lora_ranks;
  p.scalings = scalings;
  p.usorted = usorted;
  p.base_tiles = base_tiles;
  p.pieces = pieces;
  p.shrink_tiles = shrink_tiles;
  p.zgu = zgu; p.h = hbuf; p.zd = zd; p.yacc = yacc;
  p.zslice_blk = INT32_MAX;
  p.status = d_status;

  if (L > 0) {
    if (gemv_rows > 0 &&
        (rc = launch_gemv<2>(gemv_tiles, counts + 2, f.max_gemv, lora_a_gu, xs, H, f, E, R, lora_ranks, scalings,
                             zgu, stream)) != MLR_OK)
      return rc;
    Params q = p;
    q.n_tiles = counts + 1; q.nblk = f.mtiles_gu; q.abox_mask = abox_gu; q.a3_mask = a3_gu; q.aw_mask = aw_gu;
    q.rmask = rm_sgu;
    if ((rc = launch_gemm<kShrinkGU>(m_sgu, q, f.max_shrink, stream)) != MLR_OK) return rc;
  }
  prof_mark(prof, 2, stream);
  {
    Params q = p;
    // a CTA pair covers 256 rows of I (bf16), a single CTA 128
    q.n_tiles = counts; q.nblk = (int)ceil_div(I, qf == kQNone ? 256 : 128); q.rmask = rm_gu; q.w3 = w3;
    q.wscale = s_gu; q.wzero = z_gu; q.wsr = (int)ceil_div(2 * I, 128); q.wsc = (int)ceil_div(H, 128);
    q.wexp = z_gu; q.sfx = sx; q.h8 = h8; q.sh = sh;
    rc = qf == kQFp8 ? launch_gemm<kGateUp, kQFp8>(m_gu, q, f.max_base, stream)
       : qf == kQMx ? launch_gemm<kGateUp, kQMx>(m_gu, q, f.max_base, stream)
       : qf == kQInt8 ? launch_gemm<kGateUp, kQInt8>(m_gu, q, f.max_base, stream)
       : qf == kQU4 ? launch_gemm<kGateUp, kQU4>(m_gu, q, f.max_base, stream)
                    : launch_gemm<kGateUp>(m_gu, q, f.max_base, stream);
    if (rc != MLR_OK) return rc;
  }
  prof_mark(prof, 3, stream);
  if (L > 0) {
    if (gemv_rows > 0 &&
        (rc = launch_gemv<1>(gemv_tiles, counts + 2, f.max_gemv, lora_a_down, hbuf, I, f, E, R, lora_ranks,
                             scalings, zd, stream)) != MLR_OK)
      return rc;
    Params q = p;
    q.n_tiles = counts + 1; q.nblk = f.mtiles_d; q.abox_mask = abox_d; q.aw_mask = aw_d; q.rmask = rm_sd;
    if ((rc = launch_gemm<kShrinkD>(m_sd, q, f.max_shrink, stream)) != MLR_OK) return rc;
  }
  prof_mark(prof, 4, stream);
  {
    Params q = p;
    // a CTA pair covers 256 rows of H (bf16), a single CTA 128 (weights
    // dequantised on chip) or two blocks of 128 (block-scaled FP8)
    q.n_tiles = counts; q.nblk = (int)ceil_div(H, quant && !mx ? 128 : 256); q.rmask = rm_dn;
    q.ykeep = (int64_t)T * H * 4 <= ((int64_t)64 << 20) ? 1 : 0;  // half of the 129 MB L2
    q.dpair = det ? xs : nullptr;
    q.wscale = s_d; q.wzero = z_d; q.wsr = (int)ceil_div(H, 128); q.wsc = (int)ceil_div(I, 128);
    q.wexp = z_d; q.sfx = sh;
    rc = qf == kQFp8 ? launch_gemm<kDown, kQFp8>(m_dn, q, f.max_base, stream)
       : qf == kQMx ? launch_gemm<kDown, kQMx>(m_dn, q, f.max_base, stream)
       : qf == kQInt8 ? launch_gemm<kDown, kQInt8>(m_dn, q, f.max_base, stream)
       : qf == kQU4 ? launch_gemm<kDown, kQU4>(m_dn, q, f.max_base, stream)
                    : launch_gemm<kDown>(m_dn, q, f.max_base, stream);
    if (rc != MLR_OK) return rc;
  }
  prof_mark(prof, 5, stream);
  const int64_t n = (int64_t)T * H;
  {
    const cudaError_t e =
        det ? launch_pdl(combine_kernel, dim3((unsigned)ceil_div(n / 8, 256)), dim3(256), 0, stream, xs, topk_ids,
                         token_lora_mapping, T, K, H, E, L, y)
            : launch_pdl(convert_kernel, dim3((unsigned)ceil_div(ceil_div(n, 4), 256)), dim3(256), 0, stream, yacc, y, n);
    if (e != cudaSuccess) return MLR_ERR_CUDA;
  }
  MLR_CHECK_LAUNCH();
  note_launch();
  prof_mark(prof, 6, stream);
  return MLR_OK;
}

}  // namespace
}  // namespace mlr

extern "C" int fused_moe_lora_forward(const mlr_bf16* x, const int32_t* topk_ids, const float* topk_weights,
                                      const int32_t* token_lora_mapping, const int32_t* lora_ranks,
                                      const float* scalings, const mlr_bf16* w_gate_up,
                                      const mlr_bf16* w_down, const mlr_bf16* lora_a_gu,
                                      const mlr_bf16* lora_b_gu, const mlr_bf16* lora_a_down,
                                      const mlr_bf16* lora_b_down, int32_t T, int32_t K, int32_t E,
                                      int32_t H, int32_t I, int32_t L, int32_t R, mlr_bf16* y,
                                      void* workspace, size_t ws_bytes, int32_t* d_status,
                                      void* stream_) {
  return mlr::moe_forward(x, topk_ids, topk_weights, token_lora_mapping, lora_ranks, scalings, w_gate_up, w_down,
                          nullptr, nullptr, nullptr, nullptr, mlr::kQNone, lora_a_gu, lora_b_gu, lora_a_down,
                          lora_b_down, T, K, E, H, I, L, R, y, workspace, ws_bytes, d_status,
                          static_cast<cudaStream_t>(stream_));
}

extern "C" int fused_moe_lora_forward_fp8(const mlr_bf16* x, const int32_t* topk_ids,
                                          const float* topk_weights, const int32_t* token_lora_mapping,
                                          const int32_t* lora_ranks, const float* scalings,
                                          const uint8_t* w_gate_up_q, const float* w_gate_up_scale,
                                          const uint8_t* w_down_q, const float* w_down_scale,
                                          const mlr_bf16* lora_a_gu, const mlr_bf16* lora_b_gu,
                                          const mlr_bf16* lora_a_down, const mlr_bf16* lora_b_down, int32_t T,
                                          int32_t K, int32_t E, int32_t H, int32_t I, int32_t L, int32_t R,
                                          mlr_bf16* y, void* workspace, size_t ws_bytes, int32_t* d_status,
                                          void* stream_) {
  return mlr::moe_forward(x, topk_ids, topk_weights, token_lora_mapping, lora_ranks, scalings, w_gate_up_q,
                          w_down_q, w_gate_up_scale, w_down_scale, nullptr, nullptr, mlr::kQFp8, lora_a_gu,
                          lora_b_gu, lora_a_down, lora_b_down, T, K, E, H, I, L, R, y, workspace, ws_bytes,
                          d_status, static_cast<cudaStream_t>(stream_));
}

extern "C" int fused_moe_lora_forward_int8(const mlr_bf16* x, const int32_t* topk_ids,
                                           const float* topk_weights, const int32_t* token_lora_mapping,
                                           const int32_t* lora_ranks, const float* scalings,
                                           const int8_t* w_gate_up_q, const float* w_gate_up_scale,
                                           const int8_t* w_down_q, const float* w_down_scale,
                                           const mlr_bf16* lora_a_gu, const mlr_bf16* lora_b_gu,
                                           const mlr_bf16* lora_a_down, const mlr_bf16* lora_b_down, int32_t T,
                                           int32_t K, int32_t E, int32_t H, int32_t I, int32_t L, int32_t R,
                                           mlr_bf16* y, void* workspace, size_t ws_bytes, int32_t* d_status,
                                           void* stream_) {
  return mlr::moe_forward(x, topk_ids, topk_weights, token_lora_mapping, lora_ranks, scalings, w_gate_up_q,
                          w_down_q, w_gate_up_scale, w_down_scale, nullptr, nullptr, mlr::kQInt8, lora_a_gu,
                          lora_b_gu, lora_a_down, lora_b_down, T, K, E, H, I, L, R, y, workspace, ws_bytes,
                          d_status, static_cast<cudaStream_t>(stream_));
}

extern "C" int fused_moe_lora_forward_w4a16(const mlr_bf16* x, const int32_t* topk_ids,
                                            const float* topk_weights, const int32_t* token_lora_mapping,
                                            const int32_t* lora_ranks, const float* scalings,
                                            const uint8_t* w_gate_up_q, const float* w_gate_up_scale,
                                            const uint8_t* w_gate_up_zero, const uint8_t* w_down_q,
                                            const float* w_down_scale, const uint8_t* w_down_zero,
                                            const mlr_bf16* lora_a_gu, const mlr_bf16* lora_b_gu,
                                            const mlr_bf16* lora_a_down, const mlr_bf16* lora_b_down, int32_t T,
                                            int32_t K, int32_t E, int32_t H, int32_t I, int32_t L, int32_t R,
                                            mlr_bf16* y, void* workspace, size_t ws_bytes, int32_t* d_status,
                                            void* stream_) {
  return mlr::moe_forward(x, topk_ids, topk_weights, token_lora_mapping, lora_ranks, scalings, w_gate_up_q,
                          w_down_q, w_gate_up_scale, w_down_scale, w_gate_up_zero, w_down_zero, mlr::kQU4,
                          lora_a_gu, lora_b_gu, lora_a_down, lora_b_down, T, K, E, H, I, L, R, y, workspace,
                          ws_bytes, d_status, static_cast<cudaStream_t>(stream_));
}

extern "C" int fused_moe_lora_forward_fp8_w8a8(const mlr_bf16* x, const int32_t* topk_ids,
                                               const float* topk_weights, const int32_t* token_lora_mapping,
                                               const int32_t* lora_ranks, const float* scalings,
                                               const uint8_t* w_gate_up_q, const uint8_t* w_gate_up_exp,
                                               const uint8_t* w_down_q, const uint8_t* w_down_exp,
                                               const mlr_bf16* lora_a_gu, const mlr_bf16* lora_b_gu,
                                               const mlr_bf16* lora_a_down, const mlr_bf16* lora_b_down, int32_t T,
                                               int32_t K, int32_t E, int32_t H, int32_t I, int32_t L, int32_t R,
                                               mlr_bf16* y, void* workspace, size_t ws_bytes, int32_t* d_status,
                                               void* stream_) {
  return mlr::moe_forward(x, topk_ids, topk_weights, token_lora_mapping, lora_ranks, scalings, w_gate_up_q,
                          w_down_q, nullptr, nullptr, w_gate_up_exp, w_down_exp, mlr::kQMx, lora_a_gu, lora_b_gu,
                          lora_a_down, lora_b_down, T, K, E, H, I, L, R, y, workspace, ws_bytes, d_status,
                          static_cast<cudaStream_t>(stream_));
}

// ------------------------------------------------------------------------
// Dense projection with per-segment LoRA and split B (the MLA fused
// q_a_proj + kv_a_proj projection): the same machinery as one expert with
// top-1 routing.  Tokens are ordered by adapter, gathered, shrunk per adapter
// bucket (one or two rank blocks), then one GEMM on CTA pairs computes
// W x + s B z per output block, reading the rank block of the block's part.
// ------------------------------------------------------------------------
namespace mlr {
namespace {

// Workspace of the projection: the forward's layout for one expert, top-1,
// with the wider of D_in / D_out as its hidden size (x_sorted and y_acc) and
// the smallest intermediate size.
FwdLayout lin_layout(int32_t T, int32_t D_in, int32_t D_out, int32_t L, int32_t R, int32_t S) {
  FwdLayout f{};
  f.ok = false;
  if (T < 0 || D_in < 128 || D_out < 128 || D_in % 8 || D_out % 8 || (S != 1 && S != 2)) return f;
  return fwd_layout(T, 1, 1, D_in > D_out ? D_in : D_out, 64, L, R);
}

}  // namespace
}  // namespace mlr

extern "C" size_t lora_linear_workspace_bytes(int32_t num_tokens, int32_t in_features, int32_t out_features,
                                              int32_t num_loras, int32_t max_rank, int32_t num_slices) {
  const mlr::FwdLayout f = mlr::lin_layout(num_tokens, in_features, out_features, num_loras, max_rank, num_slices);
  return f.ok ? (size_t)f.total : 0;
}

extern "C" int lora_linear_forward(const mlr_bf16* x, const mlr_bf16* w, const int32_t* token_lora_mapping,
                                   const int32_t* lora_ranks, const float* scalings, const mlr_bf16* lora_a,
                                   const mlr_bf16* lora_b, const int32_t* slice_offsets, int32_t T, int32_t D_in,
                                   int32_t D_out, int32_t L, int32_t R, int32_t S, mlr_bf16* y, void* workspace,
                                   size_t ws_bytes, int32_t* d_status, void* stream_) {
  using namespace mlr;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  if (slice_offsets == nullptr || (S != 1 && S != 2)) return MLR_ERR_INVALID;
  // parts: 0 = offsets[0] < offsets[1] < ... = D_out; the second part starts on
  // a 256-row block (one output block of a CTA pair)
  if (slice_offsets[0] != 0 || slice_offsets[S] != D_out) return MLR_ERR_INVALID;
  if (S == 2 && (slice_offsets[1] <= 0 || slice_offsets[1] >= D_out || slice_offsets[1] % 256 != 0))
    return MLR_ERR_INVALID;
  const FwdLayout f = lin_layout(T, D_in, D_out, L, R, S);
  if (!f.ok) {
    if (T < 0 || L < 0 || R < 0) return MLR_ERR_INVALID;
    return MLR_ERR_UNSUPPORTED;
  }
  if (T == 0) return MLR_OK;
  const void* need[] = {x, w, token_lora_mapping, y};
  for (const void* q : need)
    if (q == nullptr) return MLR_ERR_INVALID;
  if (L > 0 && (lora_ranks == nullptr || scalings == nullptr || lora_a == nullptr || lora_b == nullptr))
    return MLR_ERR_INVALID;
  const void* aligned[] = {x, w, lora_a, lora_b, y};
  for (const void* q : aligned)
    if ((reinterpret_cast<uintptr_t>(q) & 15) != 0) return MLR_ERR_INVALID;
  if (workspace == nullptr || ws_bytes < (size_t)f.total) return MLR_ERR_CAPACITY;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255) != 0) return MLR_ERR_INVALID;

  char* ws = static_cast<char*>(workspace);
  char* aws = ws + f.o_align;
  TileRec* base_tiles = reinterpret_cast<TileRec*>(ws + f.o_base);
  ShrinkRec* shrink_tiles = reinterpret_cast<ShrinkRec*>(ws + f.o_shrink);
  ShrinkRec* gemv_tiles = reinterpret_cast<ShrinkRec*>(ws + f.o_gemv);
  int4* pieces = reinterpret_cast<int4*>(ws + f.o_pieces);
  uint32_t* ustart = reinterpret_cast<uint32_t*>(ws + f.o_ustart);
  int32_t* usorted = reinterpret_cast<int32_t*>(ws + f.o_usorted);
  int32_t* counts = reinterpret_cast<int32_t*>(ws + f.o_counts);
  uint16_t* z = reinterpret_cast<uint16_t*>(ws + (S == 2 ? f.o_zgu : f.o_zd));
  float* yacc = reinterpret_cast<float*>(ws + f.o_yacc);
  uint16_t* xs = reinterpret_cast<uint16_t*>(ws + f.o_xs);
  const uint32_t* btotal = reinterpret_cast<const uint32_t*>(aws + f.al.btotal_off);

  // tensor maps: the shrink (two rank blocks = the gate_up-shape shrink with
  // the parts as gate and up; one block = the down-shape shrink) and the
  // projection on CTA pairs
  Maps m_s{}, m_p{};
  int abox = 0, a3 = 0, aw = 0, rm = 0;
  const uint64_t cap = (uint64_t)f.cap, zcap = (uint64_t)f.zcap;
  bool ok = S == 2 ? make_shrink2_maps(m_s, xs, cap, D_in, lora_a, L, 1, R, &abox, &a3, &aw, &rm)
                   : make_shrink1_maps(m_s, xs, cap, D_in, lora_a, L, 1, R, &abox, &aw, &rm);
  ok = ok && make_down_maps(m_p, w, D_out, D_in, 1, xs, cap, lora_b, L, R, z, zcap, S * f.R16 / 8);
  if (!ok) return MLR_ERR_CUDA;

  const int prof = prof_call_begin(stream);
  int rc = MLR_OK;
  const int64_t nb_nonempty = f.al.P < f.al.NB ? f.al.P : f.al.NB;
  const int gemv_rows = (L > 0 && f.al.P < 8 * nb_nonempty) ? kGemvRows : 0;
  const size_t scan_bytes = (size_t)round_up(((int64_t)f.al.NB + 1) * 4, 16);
  int32_t* zeros_ids = reinterpret_cast<int32_t*>(ws + f.o_h);  // expert id 0 of every token
  if (cudaMemsetAsync(zeros_ids, 0, (size_t)T * 4, stream) != cudaSuccess) return MLR_ERR_CUDA;
  if (align_block_ok(f.al, scan_bytes)) {
    const size_t zs_off = align_block_smem(f.al), sm = zs_off + scan_bytes;
    if (sm > 48 * 1024 &&
        cudaFuncSetAttribute(align_plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm) != cudaSuccess)
      return MLR_ERR_CUDA;
    if (launch_pdl(align_plan_kernel, dim3(1), dim3(kPlanThreads), sm, stream, zeros_ids, token_lora_mapping, (int)f.al.P, 1, 1, L, R,
                                                       lora_ranks, usorted, ustart, base_tiles, pieces,
                                                       shrink_tiles, gemv_tiles, counts, d_status, (int)zs_off,
                                                       gemv_rows, 0, kTileRows, 0) != cudaSuccess) return MLR_ERR_CUDA;
    MLR_CHECK_LAUNCH();
    note_launch();
  } else {
    if ((rc = align_dense_count(f.al, zeros_ids, token_lora_mapping, 1, 1, L, aws, d_status, stream)) != MLR_OK)
      return rc;
    const size_t sm = 2 * scan_bytes;
    if (sm > 48 * 1024 &&
        cudaFuncSetAttribute(plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm) != cudaSuccess)
      return MLR_ERR_CUDA;
    if (launch_pdl(plan_kernel, dim3(1), dim3(kPlanThreads), sm, stream, btotal, lora_ranks, 1, f.C, R, ustart, base_tiles, pieces,
                                                  shrink_tiles, gemv_tiles, counts, d_status, gemv_rows, 0,
                                                  kTileRows, 0) != cudaSuccess) return MLR_ERR_CUDA;
    MLR_CHECK_LAUNCH();
    note_launch();
    if ((rc = align_dense_scatter(f.al, zeros_ids, token_lora_mapping, 1, 1, L, aws, ustart, usorted, stream)) !=
        MLR_OK)
      return rc;
  }
  prof_mark(prof, 0, stream);
  {
    const int64_t blocks = ceil_div(f.cap, kGatherThreads / 32);
    const int grid = (int)(blocks < 16 * sm_count() ? blocks : 16 * sm_count());
    if (launch_pdl(gather_x_kernel, dim3(grid), dim3(kGatherThreads), 0, stream, x, usorted, ustart + f.al.NB, 1, D_in, f.cap, xs, yacc,
                                                         (int64_t)T * D_out / 4) != cudaSuccess) return MLR_ERR_CUDA;
    MLR_CHECK_LAUNCH();
    note_launch();
  }
  prof_mark(prof, 1, stream);

  Params p{};
  p.T = T; p.K = 1; p.E = 1; p.L = L; p.R = R; p.R16 = f.R16; p.C = f.C;
  p.cap = (int)f.cap;
  p.zcap = (int)f.zcap;
  p.zrows = (int)(f.zcap < 256 ? f.zcap : 256);
  p.zshort = p.zrows >= 64 ? 1 : 0;
  p.bmask = L > 0 ? b_view_mask(R) : 0;
  p.P = T;
  p.wait_ns = wait_limit_ns();
  p.topk_weights = nullptr;  // weight 1 for every token
  p.lora_ranks = lora_ranks;
  p.scalings = scalings;
  p.usorted = usorted;
  p.base_tiles = base_tiles;
  p.pieces = pieces;
  p.shrink_tiles = shrink_tiles;
  p.yacc = yacc;
  p.status = d_status;
  p.zslice_blk = S == 2 ? slice_offsets[1] / 256 : INT32_MAX;
  if (L > 0) {
    Params q = p;
    q.n_tiles = counts + 1; q.abox_mask = abox; q.aw_mask = aw; q.rmask = rm;
    if (S == 2) {
      // the parts' A blocks stand where gate_up's gate and up blocks stand
      q.H = D_in; q.nblk = f.mtiles_gu; q.a3_mask = a3; q.zgu = z;
      if (gemv_rows > 0 &&
          (rc = launch_gemv<2>(gemv_tiles, counts + 2, f.max_gemv, lora_a, xs, D_in, f, 1, R, lora_ranks,
                               scalings, z, stream)) != MLR_OK)
        return rc;
      if ((rc = launch_gemm<kShrinkGU>(m_s, q, f.max_shrink, stream)) != MLR_OK) return rc;
    } else {
      q.I = D_in; q.nblk = f.mtiles_d; q.zd = z;
      if (gemv_rows > 0 &&
          (rc = launch_gemv<1>(gemv_tiles, counts + 2, f.max_gemv, lora_a, xs, D_in, f, 1, R, lora_ranks,
                               scalings, z, stream)) != MLR_OK)
        return rc;
      if ((rc = launch_gemm<kShrinkD>(m_s, q, f.max_shrink, stream)) != MLR_OK) return rc;
    }
  }
  prof_mark(prof, 2, stream);
  prof_mark(prof, 3, stream);
  prof_mark(prof, 4, stream);
  {
    Params q = p;
    q.H = D_out; q.I = D_in;  // output rows and K of the down-shape GEMM
    q.n_tiles = counts; q.nblk = (int)ceil_div(D_out, 256);
    q.ykeep = (int64_t)T * D_out * 4 <= ((int64_t)64 << 20) ? 1 : 0;
    if ((rc = launch_gemm<kDown>(m_p, q, f.max_base, stream)) != MLR_OK) return rc;
  }
  prof_mark(prof, 5, stream);
  const int64_t n = (int64_t)T * D_out;
  if (launch_pdl(convert_kernel, dim3((unsigned)ceil_div(ceil_div(n, 4), 256)), dim3(256), 0, stream, yacc, y, n) != cudaSuccess) return MLR_ERR_CUDA;
  MLR_CHECK_LAUNCH();
  note_launch();
  prof_mark(prof, 6, stream);
  return MLR_OK;
}
