/*
 * moe_lora_oracle.c -- plain, slow, obviously-correct CPU oracle for the
 * multi-adapter LoRA mixture-of-experts expert layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file: only the test-suite, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header, table or helper with
 * the CUDA library under lora_moe_expert_info_gb300/csrc.
 *
 * Sources (web pages summarising sglang pull requests):
 *   [PR14105] "LoRA on MoE expert layers" page, section 实现拆解 (implementation
 *             breakdown): the layer formula
 *               y = (W_down + a/r B_d A_d)[SiLU((W_gate + a/r B_g A_g)x)
 *                                          (.) ((W_up + a/r B_u A_u)x)],
 *             the align kernel that orders tokens by LoRA adapter and expert
 *             id, and the 4-D adapter stack [num_loras, num_experts, rank, dim].
 *   [PR22323] "LoRA quantisation info and DeepSeek-V3 MLA fused projection"
 *             page, section 实现拆解 items 2-3: ReplicatedLinearWithLoRA applies
 *             LoRA to the fused q_a_proj + kv_a_proj_with_mqa projection, its B
 *             split into two parts applied by two segment GEMMs.  Its 功能与动机
 *             section and 实现拆解 item 1: quantised MoE experts (FP8,
 *             block-wise INT8, WNA16) hand their scales to the LoRA MoE layer,
 *             which then runs with quantised base weights.
 *   [PR24160] "shared MoE LoRA batch info" page, sections 实现拆解 and
 *             关键源码片段 (MoELoRABatchInfo dataclass; test_moe_lora_info.py):
 *             token_lora_mapping = repeat_interleave(weight_indices, seg_lens),
 *             adapter_enabled = scatter of (rank > 0) at weight_indices, -1 means
 *             "no adapter", and the "under-covers tokens" launch check.
 *
 * Precision: every floating-point sum is accumulated in double.  bf16 inputs
 * are widened exactly (a bf16 value is the top 16 bits of a float).
 *
 * Readings taken where the pages are silent (each also listed in the design
 * notes):
 *   - weight_indices == -1 copies -1 into the mapping and never touches
 *     adapter_enabled; slots no request uses are 0.
 *   - align key order is expert-major, adapter-minor, with "no adapter" (-1)
 *     first inside each expert; ties keep ascending pair index p = t*K + k.
 *     Every non-empty bucket is padded to a multiple of block_size with the
 *     sentinel P = T*K.
 *   - the top-k weight multiplies the whole expert output, LoRA delta
 *     included; an adapter contributes iff its id is >= 0 and its rank > 0;
 *     only the first rank columns/rows of the zero-padded stacks are read.
 *   - quantised experts (the pages name the methods, not their formats): FP8
 *     E4M3 expert weights, each 128 x 128 block (rows x columns of W_gate_up
 *     [E, 2I, H] and W_down [E, H, I]) with one float scale, the weight being
 *     code value x scale (the DeepSeek-V3 checkpoint layout, inverse scales
 *     [E, ceil(rows/128), ceil(cols/128)]).  Activations, LoRA A and B stay
 *     bf16; only the base weights are quantised.
 *   - FP8 on FP8 tensor cores (W8A8, MX-style scaling): E4M3 expert weights
 *     whose 128 x 128 block scales are powers of two, stored as biased 8-bit
 *     exponents (UE8M0: scale = 2^(e - 127)); the activations that feed the
 *     base GEMMs are quantised too, per token and group of 128 channels, with
 *     a power-of-two scale 2^s, s the smallest integer with
 *     max|group| x 2^-s <= 448 (clamped to [-127, 127]; 0 for an all-zero
 *     group), each element rounded to the nearest E4M3 value (ties to even).
 *     x is quantised from its bf16 value; the intermediate a = SiLU(g) * u is
 *     first rounded to bf16 (the stored intermediate) and then quantised the
 *     same way for the down GEMM.  The LoRA shrinks read the unquantised
 *     (bf16) x and a.  Since a's quantisation (an integer decision) depends
 *     on the LoRA delta, this layer takes it at the kernels' precision: the
 *     scaled LoRA intermediates s_l * (A x) and s_l * (A_d a) are rounded to
 *     bf16 before B multiplies them, as the GPU stores them.
 *
 * Parity pins (see tests/test_oracle_*.py): the worked mapping example of
 * [PR24160]; torch.repeat_interleave on random segments; brute-force sorted()
 * for align; a dense SwiGLU MLP via torch for one expert; dense-materialised
 * W + s*B*A against the factored form; base identity for B = 0, adapter -1
 * and rank 0; linearity and permutation invariances of the top-k combine;
 * for FP8 experts, the E4M3 decoder against the format's defining values and
 * torch's float8_e4m3fn for all 256 codes, and the layer against the fp64
 * forward on weights dequantised with numpy (unit and power-of-two block
 * scales, ragged and gate/up-shared blocks); for the W8A8 layer, the E4M3
 * rounding against torch's float8 cast on every tie, the group exponent
 * against ceil(log2(amax / 448)), and the layer against a torch float64
 * re-derivation with planted mistakes that must change it.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_OK 0
#define ORC_INVALID (-1)
#define ORC_UNDERCOVERED (-2)
#define ORC_INDEX (-3)
#define ORC_CAPACITY (-4)
#define ORC_NOMEM (-7)

/* ------------------------------------------------------------------------ */
/* batch info  ([PR24160] 实现拆解 items 1-3; 关键源码片段: dataclass fields and  */
/* the expected-value rules of test_compute_moe_lora_info_expands_segments)  */
/* ------------------------------------------------------------------------ */

/*
 * seg_indptr[bs+1], weight_indices[bs], lora_ranks[num_loras]
 *   -> token_lora_mapping[num_tokens], adapter_enabled[num_loras].
 * max_len > 0 is the launch hint of the page's kernel: a launch of bs segments
 * of at most max_len tokens each under-covers the batch when
 * bs * max_len < num_tokens or some segment is longer than max_len.
 */
int oracle_batch_info(const int32_t* seg_indptr, const int32_t* weight_indices,
                      const int32_t* lora_ranks, int32_t bs, int32_t num_loras,
                      int32_t num_tokens, int32_t max_len,
                      int32_t* token_lora_mapping, int32_t* adapter_enabled) {
  if (bs < 0 || num_loras < 0 || num_tokens < 0 || max_len < 0) return ORC_INVALID;
  if (seg_indptr[0] != 0 || seg_indptr[bs] != num_tokens) return ORC_INVALID;
  for (int32_t i = 0; i < bs; ++i)
    if (seg_indptr[i + 1] < seg_indptr[i]) return ORC_INVALID;
  if (max_len > 0) {
    if ((int64_t)bs * (int64_t)max_len < (int64_t)num_tokens) return ORC_UNDERCOVERED;
    for (int32_t i = 0; i < bs; ++i)
      if (seg_indptr[i + 1] - seg_indptr[i] > max_len) return ORC_UNDERCOVERED;
  }
  for (int32_t i = 0; i < bs; ++i)
    if (weight_indices[i] < -1 || weight_indices[i] >= num_loras) return ORC_INDEX;

  /* token_lora_mapping: request i's adapter repeated over its segment. */
  for (int32_t i = 0; i < bs; ++i)
    for (int32_t t = seg_indptr[i]; t < seg_indptr[i + 1]; ++t)
      token_lora_mapping[t] = weight_indices[i];

  /* adapter_enabled: zeros, then 1 at each used slot whose rank is > 0. */
  for (int32_t l = 0; l < num_loras; ++l) adapter_enabled[l] = 0;
  for (int32_t i = 0; i < bs; ++i) {
    int32_t l = weight_indices[i];
    if (l >= 0) adapter_enabled[l] = (lora_ranks[l] > 0) ? 1 : 0;
  }
  return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* (lora, expert) align  ([PR14105] 实现拆解: the align kernel sorts tokens by  */
/* LoRA adapter and expert id; block_size padding as in the page's name)     */
/* ------------------------------------------------------------------------ */

/* Upper bound on the padded length: every non-empty bucket adds < block_size. */
int64_t oracle_align_capacity(int32_t num_tokens, int32_t topk, int32_t num_experts,
                              int32_t num_loras, int32_t block_size) {
  if (num_tokens < 0 || topk < 1 || num_experts < 1 || num_loras < 0 || block_size < 1)
    return -1;
  int64_t P = (int64_t)num_tokens * topk;
  int64_t NB = (int64_t)num_experts * (num_loras + 1);
  int64_t buckets = P < NB ? P : NB;
  int64_t n = P + buckets * (block_size - 1);
  return (n + block_size - 1) / block_size * block_size;
}

/*
 * topk_ids[T*K] (expert of pair p = t*K + k), token_lora_mapping[T]
 *   -> sorted_token_ids[capacity] (pair ids; pad slots hold P),
 *      block_expert_ids[capacity/block_size], block_lora_ids[...],
 *      *num_tokens_post_pad.
 * A stable counting sort on key = e*(L+1) + (lora+1).
 */
int oracle_align(const int32_t* topk_ids, const int32_t* token_lora_mapping,
                 int32_t num_tokens, int32_t topk, int32_t num_experts, int32_t num_loras,
                 int32_t block_size, int32_t* sorted_token_ids, int32_t* block_expert_ids,
                 int32_t* block_lora_ids, int32_t* num_tokens_post_pad, int64_t capacity) {
  if (num_tokens < 0 || topk < 1 || num_experts < 1 || num_loras < 0 || block_size < 1)
    return ORC_INVALID;
  const int64_t P = (int64_t)num_tokens * topk;
  if (P >= INT32_MAX) return ORC_INVALID;
  const int64_t C = (int64_t)num_loras + 1;      /* adapter classes per expert */
  const int64_t NB = (int64_t)num_experts * C;   /* buckets                    */

  int64_t* count = (int64_t*)calloc((size_t)NB, sizeof(int64_t));
  int64_t* start = (int64_t*)calloc((size_t)NB, sizeof(int64_t));
  int64_t* cursor = (int64_t*)calloc((size_t)NB, sizeof(int64_t));
  if (!count || !start || !cursor) {
    free(count); free(start); free(cursor);
    return ORC_NOMEM;
  }

  /* 1. count pairs per bucket, rejecting ids outside their ranges */
  for (int64_t p = 0; p < P; ++p) {
    int32_t e = topk_ids[p];
    int32_t l = token_lora_mapping[p / topk];
    if (e < 0 || e >= num_experts || l < -1 || l >= num_loras) {
      free(count); free(start); free(cursor);
      return ORC_INDEX;
    }
    count[(int64_t)e * C + (l + 1)] += 1;
  }

  /* 2. bucket starts: exclusive running sum of counts rounded up to block_size */
  int64_t total = 0;
  for (int64_t b = 0; b < NB; ++b) {
    start[b] = total;
    total += (count[b] + block_size - 1) / block_size * block_size;
  }
  if (total > capacity) {
    free(count); free(start); free(cursor);
    return ORC_CAPACITY;
  }

  /* 3. place pairs in increasing p: stable within a bucket */
  for (int64_t b = 0; b < NB; ++b) cursor[b] = start[b];
  for (int64_t p = 0; p < P; ++p) {
    int64_t b = (int64_t)topk_ids[p] * C + (token_lora_mapping[p / topk] + 1);
    sorted_token_ids[cursor[b]] = (int32_t)p;
    cursor[b] += 1;
  }

  /* 4. pad each bucket's tail with the sentinel P; label its blocks */
  for (int64_t b = 0; b < NB; ++b) {
    int64_t padded = (count[b] + block_size - 1) / block_size * block_size;
    for (int64_t j = count[b]; j < padded; ++j) sorted_token_ids[start[b] + j] = (int32_t)P;
    for (int64_t blk = start[b] / block_size; blk < (start[b] + padded) / block_size; ++blk) {
      block_expert_ids[blk] = (int32_t)(b / C);
      block_lora_ids[blk] = (int32_t)(b % C) - 1;
    }
  }
  *num_tokens_post_pad = (int32_t)total;

  free(count); free(start); free(cursor);
  return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* forward  ([PR14105] 实现拆解: FusedMoEWithLoRA formula; top-k weighted sum  */
/* over the selected experts; 4-D stacks [num_loras, num_experts, rank, dim]) */
/* ------------------------------------------------------------------------ */

/* dtype 0: bf16 bit patterns (uint16); dtype 1: IEEE double. */
static double ld(const void* base, int dtype, int64_t idx) {
  if (dtype == 0) {
    uint32_t u = (uint32_t)((const uint16_t*)base)[idx] << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
  }
  return ((const double*)base)[idx];
}

static double silu(double z) { return z / (1.0 + exp(-z)); }

/*
 * FP8 E4M3 (the OCP 8-bit floating-point format's E4M3 encoding, as used for
 * DeepSeek-V3's FP8 weights): sign bit, 4 exponent bits with bias 7, 3
 * mantissa bits.  Exponent field 0 holds subnormals 0.m x 2^-6; there are no
 * infinities, and exponent and mantissa fields both all ones is NaN.  Largest
 * finite value 1.75 x 2^8 = 448.
 */
double oracle_e4m3_value(uint32_t code) {
  const int sign = (int)((code >> 7) & 1u), ef = (int)((code >> 3) & 15u), mf = (int)(code & 7u);
  double v;
  if (ef == 15 && mf == 7) return NAN;
  if (ef == 0) v = ldexp((double)mf / 8.0, -6);
  else v = ldexp(1.0 + (double)mf / 8.0, ef - 7);
  return sign ? -v : v;
}

/*
 * A base expert weight [E, rows, cols]: dtype 0 bf16 bits, 1 double,
 *   2 FP8 E4M3 codes: value = code x scale[e][row / 128][col / 128];
 *   3 INT8 codes (two's complement, -128..127): the same 128 x 128 block scales;
 *   4 UINT4 codes, two per byte along a row (element 2j in the low nibble of
 *     byte j, element 2j+1 in the high nibble), with a scale and a zero point
 *     (0..15) per row and group of 128 columns:
 *     value = (code - zero[e][row][col / 128]) x scale[e][row][col / 128].
 *   5 FP8 E4M3 codes with power-of-two block scales given as biased exponents:
 *     value = code x 2^(ex[e][row / 128][col / 128] - 127).
 */
typedef struct {
  const void* p;
  int dtype;
  const float* scale;
  int64_t rows, cols;
  const uint8_t* zero;  /* dtype 4: zero points; dtype 5: block exponents */
} WeightView;

static double ld_w(const WeightView* v, int64_t e, int64_t row, int64_t col) {
  const int64_t idx = (e * v->rows + row) * v->cols + col;
  if (v->dtype == 2 || v->dtype == 3) {
    const int64_t rb = (v->rows + 127) / 128, cb = (v->cols + 127) / 128;
    const double sc = (double)v->scale[(e * rb + row / 128) * cb + col / 128];
    const uint8_t code = ((const uint8_t*)v->p)[idx];
    if (v->dtype == 2) return oracle_e4m3_value(code) * sc;
    return (double)(code < 128 ? (int)code : (int)code - 256) * sc;
  }
  if (v->dtype == 5) {
    const int64_t rb = (v->rows + 127) / 128, cb = (v->cols + 127) / 128;
    const int ex = (int)v->zero[(e * rb + row / 128) * cb + col / 128];
    return ldexp(oracle_e4m3_value(((const uint8_t*)v->p)[idx]), ex - 127);
  }
  if (v->dtype == 4) {
    const int64_t gpr = (v->cols + 127) / 128;  /* groups per row */
    const uint8_t byte = ((const uint8_t*)v->p)[(e * v->rows + row) * (v->cols / 2) + col / 2];
    const int code = (col % 2 == 0) ? (byte & 15) : (byte >> 4);
    const int64_t g = (e * v->rows + row) * gpr + col / 128;
    return (double)(code - (int)v->zero[g]) * (double)v->scale[g];
  }
  return ld(v->p, v->dtype, idx);
}

/*
 * The nearest E4M3 value to v (ties to even), for |v| <= 448: normal values
 * 2^e x 1.mmm (e >= -6) are spaced 2^(e-3); below 2^-6 the subnormals are
 * spaced 2^-9.  rint rounds to nearest, ties to even.
 */
double oracle_e4m3_round(double v) {
  const double a = fabs(v);
  if (a == 0.0) return v;
  int E;
  frexp(a, &E);          /* a in [2^(E-1), 2^E) */
  int e = E - 1;
  if (e < -6) e = -6;
  const double step = ldexp(1.0, e - 3);
  const double q = rint(a / step) * step;
  return v < 0.0 ? -q : q;
}

/*
 * The power-of-two scale exponent of a group whose largest magnitude is amax:
 * the smallest integer s with amax x 2^-s <= 448, clamped to [-127, 127];
 * 0 for amax == 0.
 */
int oracle_mx_group_exp(double amax) {
  if (!(amax > 0.0)) return 0;
  int E;
  frexp(amax, &E);
  int s = E - 9;  /* amax x 2^-s in [2^8, 2^9) */
  while (ldexp(amax, -s) > 448.0) ++s;
  while (ldexp(amax, -(s - 1)) <= 448.0) --s;
  if (s < -127) s = -127;
  if (s > 127) s = 127;
  return s;
}

/* The nearest bf16 value to v (ties to even): 8 significant bits, spacing
 * 2^-133 below 2^-126. */
static double bf16_round(double v) {
  const double a = fabs(v);
  if (a == 0.0) return v;
  int E;
  frexp(a, &E);
  int e = E - 1;
  if (e < -126) e = -126;
  const double step = ldexp(1.0, e - 7);
  const double q = rint(a / step) * step;
  return v < 0.0 ? -q : q;
}

/* q[0..n) = v quantised per group of 128 consecutive elements (the last group
 * may be shorter) and dequantised: E4M3(v x 2^-s) x 2^s, s from the group's
 * largest magnitude. */
static void quant_groups(const double* v, double* q, int64_t n) {
  for (int64_t g0 = 0; g0 < n; g0 += 128) {
    const int64_t g1 = g0 + 128 < n ? g0 + 128 : n;
    double amax = 0.0;
    for (int64_t i = g0; i < g1; ++i)
      if (fabs(v[i]) > amax) amax = fabs(v[i]);
    const int s = oracle_mx_group_exp(amax);
    for (int64_t i = g0; i < g1; ++i) q[i] = ldexp(oracle_e4m3_round(ldexp(v[i], -s)), s);
  }
}

/*
 * Layouts (row-major):
 *   x           [T, H]
 *   topk_ids    [T, K] int32, topk_weights [T, K] float
 *   mapping     [T] int32 in [-1, L);  lora_ranks [L] int32; scalings [L] float
 *   w_gate_up   [E, 2I, H]   rows 0..I-1 gate, I..2I-1 up
 *   w_down      [E, H, I]
 *   lora_a_gu   [L, E, 2, R, H]   index 0 = gate, 1 = up
 *   lora_b_gu   [L, E, 2, I, R]
 *   lora_a_down [L, E, R, I]
 *   lora_b_down [L, E, H, R]
 *   y           [n_out, H] double, row j for token tokens[j] (or j if tokens == NULL)
 */
static int forward_impl(const void* x, int x_dtype, const int32_t* topk_ids,
                        const float* topk_weights, const int32_t* token_lora_mapping,
                        const int32_t* lora_ranks, const float* scalings,
                        const WeightView* wgu, const WeightView* wdn, const void* lora_a_gu,
                        const void* lora_b_gu, const void* lora_a_down, const void* lora_b_down,
                        int w_dtype, int64_t T, int64_t K, int64_t E, int64_t H, int64_t I,
                        int64_t L, int64_t R, const int64_t* tokens, int64_t n_out, double* y,
                        int num_threads, int act_q) {
  if (T < 0 || K < 1 || E < 1 || H < 1 || I < 1 || L < 0 || R < 0 || n_out < 0)
    return ORC_INVALID;
  for (int64_t l = 0; l < L; ++l)
    if (lora_ranks[l] < 0 || lora_ranks[l] > R) return ORC_INVALID;
  for (int64_t j = 0; j < n_out; ++j) {
    int64_t t = tokens ? tokens[j] : j;
    if (t < 0 || t >= T) return ORC_INVALID;
    if (token_lora_mapping[t] < -1 || token_lora_mapping[t] >= L) return ORC_INDEX;
    for (int64_t k = 0; k < K; ++k)
      if (topk_ids[t * K + k] < 0 || topk_ids[t * K + k] >= E) return ORC_INDEX;
  }
  int status = ORC_OK;
#ifdef _OPENMP
  if (num_threads > 0) omp_set_num_threads(num_threads);
#else
  (void)num_threads;
#endif

#pragma omp parallel
  {
    double* xv = (double*)malloc(sizeof(double) * (size_t)H);
    double* a = (double*)malloc(sizeof(double) * (size_t)I);
    double* zg = (double*)malloc(sizeof(double) * (size_t)(R > 0 ? R : 1));
    double* zu = (double*)malloc(sizeof(double) * (size_t)(R > 0 ? R : 1));
    double* zd = (double*)malloc(sizeof(double) * (size_t)(R > 0 ? R : 1));
    /* act_q: the quantised x and a that feed the base GEMMs */
    double* xq = (double*)malloc(sizeof(double) * (size_t)H);
    double* aq = (double*)malloc(sizeof(double) * (size_t)I);
    const int ok = xv && a && zg && zu && zd && xq && aq;
#pragma omp for schedule(dynamic, 1)
    for (int64_t j = 0; j < n_out; ++j) {
      if (!ok) {
#pragma omp atomic write
        status = ORC_NOMEM;
        continue;
      }
      {
        const int64_t t = tokens ? tokens[j] : j;
        double* yrow = y + j * H;
        for (int64_t h = 0; h < H; ++h) yrow[h] = 0.0;
        for (int64_t h = 0; h < H; ++h) xv[h] = ld(x, x_dtype, t * H + h);
        if (act_q) quant_groups(xv, xq, H);
        const double* xb = act_q ? xq : xv;  /* the base GEMMs' input */

        const int32_t l = token_lora_mapping[t];
        const int used = (l >= 0) && (lora_ranks[l] > 0);
        const int64_t r = used ? lora_ranks[l] : 0;
        const double s = used ? (double)scalings[l] : 0.0;

        for (int64_t k = 0; k < K; ++k) {
          const int64_t e = topk_ids[t * K + k];
          const double w = (double)topk_weights[t * K + k];

          /* LoRA shrink for gate and up: z = A x (first r rows only); act_q:
           * s * z rounded to bf16 (s is then not applied again below) */
          for (int64_t q = 0; q < r; ++q) {
            const int64_t ag = (((l * E + e) * 2 + 0) * R + q) * H;
            const int64_t au = (((l * E + e) * 2 + 1) * R + q) * H;
            double sg = 0.0, su = 0.0;
            for (int64_t h = 0; h < H; ++h) {
              sg += ld(lora_a_gu, w_dtype, ag + h) * xv[h];
              su += ld(lora_a_gu, w_dtype, au + h) * xv[h];
            }
            zg[q] = act_q ? bf16_round(s * sg) : sg;
            zu[q] = act_q ? bf16_round(s * su) : su;
          }
          const double sb = act_q ? 1.0 : s;  /* the scaling still to apply after B */

          /* gate and up projections, each with its own LoRA delta; SiLU(g) * u */
          for (int64_t i = 0; i < I; ++i) {
            double g = 0.0, u = 0.0;
            for (int64_t h = 0; h < H; ++h) {
              g += ld_w(wgu, e, i, h) * xb[h];
              u += ld_w(wgu, e, I + i, h) * xb[h];
            }
            if (r > 0) {
              const int64_t bg = (((l * E + e) * 2 + 0) * I + i) * R;
              const int64_t bu = (((l * E + e) * 2 + 1) * I + i) * R;
              double dg = 0.0, du = 0.0;
              for (int64_t q = 0; q < r; ++q) {
                dg += ld(lora_b_gu, w_dtype, bg + q) * zg[q];
                du += ld(lora_b_gu, w_dtype, bu + q) * zu[q];
              }
              g += sb * dg;
              u += sb * du;
            }
            a[i] = silu(g) * u;
          }
          /* act_q: a is stored as bf16, and the down GEMM reads it quantised */
          if (act_q) {
            for (int64_t i = 0; i < I; ++i) a[i] = bf16_round(a[i]);
            quant_groups(a, aq, I);
          }
          const double* ab = act_q ? aq : a;

          /* LoRA shrink for down: zd = A_d a */
          for (int64_t q = 0; q < r; ++q) {
            const int64_t ad = ((l * E + e) * R + q) * I;
            double sd = 0.0;
            for (int64_t i = 0; i < I; ++i) sd += ld(lora_a_down, w_dtype, ad + i) * a[i];
            zd[q] = act_q ? bf16_round(s * sd) : sd;
          }

          /* down projection with its LoRA delta, weighted into y */
          for (int64_t h = 0; h < H; ++h) {
            double d = 0.0;
            for (int64_t i = 0; i < I; ++i) d += ld_w(wdn, e, h, i) * ab[i];
            if (r > 0) {
              const int64_t bd = ((l * E + e) * H + h) * R;
              double dd = 0.0;
              for (int64_t q = 0; q < r; ++q) dd += ld(lora_b_down, w_dtype, bd + q) * zd[q];
              d += sb * dd;
            }
            yrow[h] += w * d;
          }
        }
      }
    }
    free(xv); free(a); free(zg); free(zu); free(zd); free(xq); free(aq);
  }
  return status;
}

int oracle_forward(const void* x, int x_dtype, const int32_t* topk_ids,
                   const float* topk_weights, const int32_t* token_lora_mapping,
                   const int32_t* lora_ranks, const float* scalings,
                   const void* w_gate_up, const void* w_down, const void* lora_a_gu,
                   const void* lora_b_gu, const void* lora_a_down, const void* lora_b_down,
                   int w_dtype, int64_t T, int64_t K, int64_t E, int64_t H, int64_t I,
                   int64_t L, int64_t R, const int64_t* tokens, int64_t n_out, double* y,
                   int num_threads) {
  if (w_dtype != 0 && w_dtype != 1) return ORC_INVALID;
  const WeightView wgu = {w_gate_up, w_dtype, NULL, 2 * I, H, NULL};
  const WeightView wdn = {w_down, w_dtype, NULL, H, I, NULL};
  return forward_impl(x, x_dtype, topk_ids, topk_weights, token_lora_mapping, lora_ranks, scalings, &wgu,
                      &wdn, lora_a_gu, lora_b_gu, lora_a_down, lora_b_down, w_dtype, T, K, E, H, I, L, R,
                      tokens, n_out, y, num_threads, 0);
}

/*
 * The same layer with FP8 E4M3 base experts ([PR22323] 功能与动机 and 实现拆解
 * item 1: LoRA on quantised MoE models).  w_gate_up_q [E, 2I, H] and
 * w_down_q [E, H, I] hold E4M3 codes; w_gate_up_scale [E, ceil(2I/128),
 * ceil(H/128)] and w_down_scale [E, ceil(H/128), ceil(I/128)] the float scale
 * of each 128 x 128 block.  LoRA operands are bf16 bits or double (lora_dtype).
 */
int oracle_forward_fp8(const void* x, int x_dtype, const int32_t* topk_ids,
                       const float* topk_weights, const int32_t* token_lora_mapping,
                       const int32_t* lora_ranks, const float* scalings,
                       const uint8_t* w_gate_up_q, const float* w_gate_up_scale,
                       const uint8_t* w_down_q, const float* w_down_scale, const void* lora_a_gu,
                       const void* lora_b_gu, const void* lora_a_down, const void* lora_b_down,
                       int lora_dtype, int64_t T, int64_t K, int64_t E, int64_t H, int64_t I,
                       int64_t L, int64_t R, const int64_t* tokens, int64_t n_out, double* y,
                       int num_threads) {
  if (lora_dtype != 0 && lora_dtype != 1) return ORC_INVALID;
  if (w_gate_up_q == NULL || w_gate_up_scale == NULL || w_down_q == NULL || w_down_scale == NULL)
    return ORC_INVALID;
  const WeightView wgu = {w_gate_up_q, 2, w_gate_up_scale, 2 * I, H, NULL};
  const WeightView wdn = {w_down_q, 2, w_down_scale, H, I, NULL};
  return forward_impl(x, x_dtype, topk_ids, topk_weights, token_lora_mapping, lora_ranks, scalings, &wgu,
                      &wdn, lora_a_gu, lora_b_gu, lora_a_down, lora_b_down, lora_dtype, T, K, E, H, I, L,
                      R, tokens, n_out, y, num_threads, 0);
}

/*
 * The same layer with block-wise INT8 base experts ([PR22323] 功能与动机 and
 * 实现拆解 item 1 name the INT8 method, blockwise_int8): codes are signed
 * 8-bit integers with the FP8 layer's layout and 128 x 128 block scales;
 * weight = code x scale.
 */
int oracle_forward_int8(const void* x, int x_dtype, const int32_t* topk_ids,
                        const float* topk_weights, const int32_t* token_lora_mapping,
                        const int32_t* lora_ranks, const float* scalings,
                        const uint8_t* w_gate_up_q, const float* w_gate_up_scale,
                        const uint8_t* w_down_q, const float* w_down_scale, const void* lora_a_gu,
                        const void* lora_b_gu, const void* lora_a_down, const void* lora_b_down,
                        int lora_dtype, int64_t T, int64_t K, int64_t E, int64_t H, int64_t I,
                        int64_t L, int64_t R, const int64_t* tokens, int64_t n_out, double* y,
                        int num_threads) {
  if (lora_dtype != 0 && lora_dtype != 1) return ORC_INVALID;
  if (w_gate_up_q == NULL || w_gate_up_scale == NULL || w_down_q == NULL || w_down_scale == NULL)
    return ORC_INVALID;
  const WeightView wgu = {w_gate_up_q, 3, w_gate_up_scale, 2 * I, H, NULL};
  const WeightView wdn = {w_down_q, 3, w_down_scale, H, I, NULL};
  return forward_impl(x, x_dtype, topk_ids, topk_weights, token_lora_mapping, lora_ranks, scalings, &wgu,
                      &wdn, lora_a_gu, lora_b_gu, lora_a_down, lora_b_down, lora_dtype, T, K, E, H, I, L,
                      R, tokens, n_out, y, num_threads, 0);
}

/*
 * The same layer with 4-bit weights and 16-bit activations ([PR22323] names
 * the WNA16 method): w_gate_up_q [E, 2I, H/2] and w_down_q [E, H, I/2] hold
 * UINT4 codes two per byte (low nibble first); scale and zero
 * [E, rows, ceil(cols/128)] give each row's groups of 128 input columns a
 * float scale and a zero point; weight = (code - zero) x scale.  H and I even.
 */
int oracle_forward_w4a16(const void* x, int x_dtype, const int32_t* topk_ids,
                         const float* topk_weights, const int32_t* token_lora_mapping,
                         const int32_t* lora_ranks, const float* scalings,
                         const uint8_t* w_gate_up_q, const float* w_gate_up_scale,
                         const uint8_t* w_gate_up_zero, const uint8_t* w_down_q,
                         const float* w_down_scale, const uint8_t* w_down_zero, const void* lora_a_gu,
                         const void* lora_b_gu, const void* lora_a_down, const void* lora_b_down,
                         int lora_dtype, int64_t T, int64_t K, int64_t E, int64_t H, int64_t I,
                         int64_t L, int64_t R, const int64_t* tokens, int64_t n_out, double* y,
                         int num_threads) {
  if (lora_dtype != 0 && lora_dtype != 1) return ORC_INVALID;
  if (w_gate_up_q == NULL || w_gate_up_scale == NULL || w_gate_up_zero == NULL || w_down_q == NULL ||
      w_down_scale == NULL || w_down_zero == NULL || H % 2 != 0 || I % 2 != 0)
    return ORC_INVALID;
  const WeightView wgu = {w_gate_up_q, 4, w_gate_up_scale, 2 * I, H, w_gate_up_zero};
  const WeightView wdn = {w_down_q, 4, w_down_scale, H, I, w_down_zero};
  return forward_impl(x, x_dtype, topk_ids, topk_weights, token_lora_mapping, lora_ranks, scalings, &wgu,
                      &wdn, lora_a_gu, lora_b_gu, lora_a_down, lora_b_down, lora_dtype, T, K, E, H, I, L,
                      R, tokens, n_out, y, num_threads, 0);
}

/*
 * The same layer on the FP8 tensor cores (W8A8 with power-of-two block
 * scales; [PR22323] 功能与动机 and 实现拆解 item 1 name the FP8 method, the
 * format is a reading): w_gate_up_q [E, 2I, H] and w_down_q [E, H, I] hold
 * E4M3 codes; w_gate_up_exp [E, ceil(2I/128), ceil(H/128)] and w_down_exp
 * [E, ceil(H/128), ceil(I/128)] the biased exponent e of each 128 x 128
 * block (scale 2^(e - 127), e < 255).  x and the intermediate a are
 * quantised per token and 128-channel group before the base GEMMs (see the
 * readings above); the LoRA paths read them unquantised.
 */
int oracle_forward_fp8_w8a8(const void* x, int x_dtype, const int32_t* topk_ids,
                            const float* topk_weights, const int32_t* token_lora_mapping,
                            const int32_t* lora_ranks, const float* scalings,
                            const uint8_t* w_gate_up_q, const uint8_t* w_gate_up_exp,
                            const uint8_t* w_down_q, const uint8_t* w_down_exp, const void* lora_a_gu,
                            const void* lora_b_gu, const void* lora_a_down, const void* lora_b_down,
                            int lora_dtype, int64_t T, int64_t K, int64_t E, int64_t H, int64_t I,
                            int64_t L, int64_t R, const int64_t* tokens, int64_t n_out, double* y,
                            int num_threads) {
  if (lora_dtype != 0 && lora_dtype != 1) return ORC_INVALID;
  if (w_gate_up_q == NULL || w_gate_up_exp == NULL || w_down_q == NULL || w_down_exp == NULL)
    return ORC_INVALID;
  const WeightView wgu = {w_gate_up_q, 5, NULL, 2 * I, H, w_gate_up_exp};
  const WeightView wdn = {w_down_q, 5, NULL, H, I, w_down_exp};
  return forward_impl(x, x_dtype, topk_ids, topk_weights, token_lora_mapping, lora_ranks, scalings, &wgu,
                      &wdn, lora_a_gu, lora_b_gu, lora_a_down, lora_b_down, lora_dtype, T, K, E, H, I, L,
                      R, tokens, n_out, y, num_threads, 1);
}

/* ------------------------------------------------------------------------ */
/* dense projection with per-segment LoRA and split B  ([PR22323] 实现拆解   */
/* items 2-3: ReplicatedLinearWithLoRA for the fused q_a_proj +              */
/* kv_a_proj_with_mqa projection, its LoRA B split into two parts applied by */
/* two segment GEMMs, and normalize_fused_qkv_a_proj fusing the two adapter  */
/* entries into one)                                                          */
/* ------------------------------------------------------------------------ */

/*
 * The projection's output rows are split into S parts by slice_offsets[0..S]
 * (0 = slice_offsets[0] < ... < slice_offsets[S] = D_out).  Part s has its own
 * LoRA A (rank rows of A_s) and takes rows slice_offsets[s] .. slice_offsets[s+1]
 * of the stacked B.  For token t with adapter l (used iff l >= 0 and r_l > 0):
 *   y[t][o] = sum_i W[o][i] x[t][i] + s_l * sum_{q < r_l} B[l][o][q] * z_s[q],
 *   z_s[q]  = sum_i A[l][s][q][i] x[t][i],   s = the part that holds row o.
 * Layouts (row-major): x [T, D_in]; w [D_out, D_in]; lora_a [L, S, R, D_in];
 * lora_b [L, D_out, R]; y [n_out, D_out] double, row j for token tokens[j]
 * (or j if tokens == NULL).
 */
int oracle_lora_linear(const void* x, int x_dtype, const int32_t* token_lora_mapping,
                       const int32_t* lora_ranks, const float* scalings, const void* w,
                       const void* lora_a, const void* lora_b, int w_dtype, int64_t T,
                       int64_t D_in, int64_t D_out, int64_t L, int64_t R, int64_t S,
                       const int64_t* slice_offsets, const int64_t* tokens, int64_t n_out,
                       double* y, int num_threads) {
  if (T < 0 || D_in < 1 || D_out < 1 || L < 0 || R < 0 || S < 1 || n_out < 0) return ORC_INVALID;
  if (slice_offsets[0] != 0 || slice_offsets[S] != D_out) return ORC_INVALID;
  for (int64_t s = 0; s < S; ++s)
    if (slice_offsets[s + 1] <= slice_offsets[s]) return ORC_INVALID;
  for (int64_t l = 0; l < L; ++l)
    if (lora_ranks[l] < 0 || lora_ranks[l] > R) return ORC_INVALID;
  for (int64_t j = 0; j < n_out; ++j) {
    const int64_t t = tokens ? tokens[j] : j;
    if (t < 0 || t >= T) return ORC_INVALID;
    if (token_lora_mapping[t] < -1 || token_lora_mapping[t] >= L) return ORC_INDEX;
  }
  int status = ORC_OK;
#ifdef _OPENMP
  if (num_threads > 0) omp_set_num_threads(num_threads);
#else
  (void)num_threads;
#endif

#pragma omp parallel
  {
    double* xv = (double*)malloc(sizeof(double) * (size_t)D_in);
    double* z = (double*)malloc(sizeof(double) * (size_t)(S * (R > 0 ? R : 1)));
    const int ok = xv && z;
#pragma omp for schedule(dynamic, 1)
    for (int64_t j = 0; j < n_out; ++j) {
      if (!ok) {
#pragma omp atomic write
        status = ORC_NOMEM;
        continue;
      }
      const int64_t t = tokens ? tokens[j] : j;
      double* yrow = y + j * D_out;
      for (int64_t i = 0; i < D_in; ++i) xv[i] = ld(x, x_dtype, t * D_in + i);
      const int32_t l = token_lora_mapping[t];
      const int used = (l >= 0) && (lora_ranks[l] > 0);
      const int64_t r = used ? lora_ranks[l] : 0;
      const double sc = used ? (double)scalings[l] : 0.0;

      /* shrink of every part: z_s = A_s x (first r rows only) */
      for (int64_t s = 0; s < S; ++s)
        for (int64_t q = 0; q < r; ++q) {
          const int64_t a = ((l * S + s) * R + q) * D_in;
          double acc = 0.0;
          for (int64_t i = 0; i < D_in; ++i) acc += ld(lora_a, w_dtype, a + i) * xv[i];
          z[s * R + q] = acc;
        }

      /* base row plus the expand of the part that holds the row */
      int64_t s = 0;
      for (int64_t o = 0; o < D_out; ++o) {
        while (o >= slice_offsets[s + 1]) ++s;
        double acc = 0.0;
        for (int64_t i = 0; i < D_in; ++i) acc += ld(w, w_dtype, o * D_in + i) * xv[i];
        if (r > 0) {
          double d = 0.0;
          for (int64_t q = 0; q < r; ++q) d += ld(lora_b, w_dtype, (l * D_out + o) * R + q) * z[s * R + q];
          acc += sc * d;
        }
        yrow[o] = acc;
      }
    }
    free(xv);
    free(z);
  }
  return status;
}

/* Threads the OpenMP runtime would use (reported beside the CPU timing). */
int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
