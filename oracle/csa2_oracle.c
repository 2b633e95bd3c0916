/*
 * csa2_oracle.c -- plain, slow CPU oracle for the CSA2 attention layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file: only tests/, __graft_entry__.smoke() and bench.py's
 * cpu_baseline / reference leg use it.  It shares no code, header, table or
 * constant with the CUDA library; the two meet only through the seeded input
 * generator.
 *
 * Every step follows the pages' statement of the method in the pages' order,
 * in double precision, with no blocking, fusion or reordering:
 *
 *   tail layout      "SGLang 如何让 DeepSeek V4.1 Flash 的后半层只处理尾部 token"
 *                    (lab.ttaoai.cn), sec. 2.1-2.3, 2.5, 2.6 and the formula box
 *                    T = min(128,E), kept positions [S-T, S), window lower bound
 *                    S-T, visible window [max(s, i-127), i].
 *   index formats    "DeepSeek V4.1 Flash 建模" (pages.haorui.li), mixed-precision
 *                    card: indexer Q/K are MXFP4 with 32-element groups; main KV
 *                    is E4M3 with one scale per 32 channels (block-32), or, in
 *                    the card's own layout, E2M1 with one E4M3 scale per 16
 *                    channels (288 B per entry); SWA rows stay FP8.
 *   index score      same page, CSA2 and Hierarchical Sparse Indexer cards; SGLang/
 *                    Miles day-0 article (theainews.cc) sec. 2 and sec. 5 (the FP4
 *                    indexer and its TP layout: MQA-shaped, heads replicated, a
 *                    score all-reduce would be needed if heads were sharded).
 *                    Reading: s(q,j) = sum_h w[q,h] * ReLU(<Qi[q,h], Ki[j]>).
 *   visibility       CSA2 card, compressor paragraph: non-overlapping groups of m
 *                    tokens; entry j is complete, hence visible to the query at
 *                    absolute position t, once its last token m*j+m-1 <= t,
 *                    i.e. n_vis(t) = floor((t+1)/m).
 *   top-K            Hierarchical card and article sec. 2: per query the 512
 *                    highest-scoring visible compressed positions.
 *   candidate pool   Hierarchical card and article sec. 2: blocks of 8 entries,
 *                    block score = max score in the block, at most 2048 blocks,
 *                    the block holding the latest position always kept; the
 *                    filter excludes nothing when every reachable position fits.
 *   encoder replay   "DeepSeek V4.1 Flash 建模", Encoder Bounded Replay card;
 *                    article sec. 4.1 and 4.3: on a prefix hit whose SWA state
 *                    is gone, the last 128 cached tokens are processed again
 *                    with the new suffix; they rebuild SWA only, the cached
 *                    global entries are read and never rewritten, and local
 *                    attention is cut at the rebuild boundary.
 *   row cut/restore  tail page sec. 2.2 and 2.7: the per-row state entering
 *                    the late layers is cut to the tail rows, and the computed
 *                    tail rows are scattered back into the full extend layout
 *                    (the other rows are left as they were).
 *   cache writes     mixed-precision card (main KV FP8 block-32 or E2M1 with an
 *                    E4M3 scale per 16, index K MXFP4 per 32) and article sec.
 *                    5, on fusions that keep the quantisation semantics: a
 *                    fused quantise-and-write keeps the rounding sequence of
 *                    the unfused one.  Reading: the
 *                    group scale is computed in fp32, x / scale in fp32, and
 *                    the element rounds to nearest (ties to even) with
 *                    saturation at the format's largest finite value.
 *   attention        article sec. 1: each query attends to its own 128-token
 *                    window and to at most 512 selected compressed positions;
 *                    one softmax over both sets; the 512-dim latent row is both
 *                    key and value (pages.haorui.li mixed-precision card).
 *
 * Readings where the pages are silent are listed in the design notes of the
 * repository; the ones that change arithmetic are restated at each function.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* data-error bits (the oracle's own copy of the library's documented values) */
enum {
  OR_ERR_RANGE_IDX = 1,
  OR_ERR_RANGE_WINDOW = 2,
  OR_ERR_RANGE_CTX = 4,
  OR_ERR_SCALE = 8,
  OR_ERR_LD = 16,
  OR_ERR_CAPACITY = 32,
  OR_ERR_BAD_EXTEND = 64,
  OR_ERR_RANGE_ROW = 256,
  OR_ERR_NONFINITE = 512
};

typedef struct {
  int32_t num_q, num_req, ratio, pad_;
  const int32_t *q_req;
  const int64_t *q_pos;
  const int64_t *kv_start, *kv_len;
  const int64_t *swa_start, *swa_pos0, *swa_len;
} oracle_batch;

/* ------------------------------------------------------------------------ */
/* Storage formats                                                           */
/* ------------------------------------------------------------------------ */

/* E2M1 (OCP Microscaling Formats v1.0): sign, 2 exponent bits with bias 1,
 * 1 mantissa bit; exponent field 0 is subnormal (0 or 0.5).  No inf / NaN. */
double oracle_e2m1_value(int code) {
  int s = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
  double mag = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
  return s ? -mag : mag;
}

/* E4M3 "FN" (OCP 8-bit Floating Point spec): sign, 4 exponent bits with bias 7,
 * 3 mantissa bits; exponent field 0 is subnormal; S.1111.111 is NaN; no inf. */
double oracle_e4m3_value(int code) {
  int s = (code >> 7) & 1, e = (code >> 3) & 15, m = code & 7;
  if (e == 15 && m == 7) return NAN;
  double mag = (e == 0) ? ldexp(m / 8.0, -6) : ldexp(1.0 + m / 8.0, e - 7);
  return s ? -mag : mag;
}

/* Element d of an MXFP4 row: the byte d/2 holds element 2i in its low nibble
 * and element 2i+1 in its high nibble; one fp32 scale per 32 elements. */
static double mxfp4_elem(const uint8_t *codes, const float *scales, int d) {
  int byte = codes[d / 2];
  int nib = (d & 1) ? (byte >> 4) : (byte & 15);
  return oracle_e2m1_value(nib) * (double)scales[d / 32];
}

/* Element d of an FP8 block-32 row. */
static double fp8_elem(const uint8_t *codes, const float *scales, int d) {
  return oracle_e4m3_value(codes[d]) * (double)scales[d / 32];
}

/* Element d of an FP4 main-KV row ("DeepSeek V4.1 Flash 建模", mixed-precision
 * card, Main KV row: E2M1 data, one E4M3 scale per 16 channels, no second-level
 * global scale; 512 x (0.5 + 1/16) = 288 B per entry).  Byte d/2 holds element
 * 2i in its low nibble and element 2i+1 in its high nibble (as the index rows). */
static double fp4kv_elem(const uint8_t *codes, const uint8_t *sf, int d) {
  int byte = codes[d / 2];
  int nib = (d & 1) ? (byte >> 4) : (byte & 15);
  return oracle_e2m1_value(nib) * oracle_e4m3_value(sf[d / 16]);
}

/* Round x to the nearest code of a sign-magnitude format whose non-negative
 * codes 0..max_code have increasing values val(c): the nearest magnitude by
 * brute force, a tie going to the code with an even last bit; magnitudes
 * beyond val(max_code) saturate to it.  The sign bit is copied from x (a
 * negative value that rounds to zero keeps its sign), as IEEE rounding does. */
static int encode_nearest(double x, int max_code, int sign_shift, double (*val)(int)) {
  const int neg = signbit(x) ? 1 : 0;
  const double a = fabs(x);
  int best = max_code;
  if (a < val(max_code)) {
    double bd = INFINITY;
    for (int c = 0; c <= max_code; ++c) {
      const double d = fabs(val(c) - a);
      if (d < bd || (d == bd && (c & 1) == 0)) {
        bd = d;
        best = c;
      }
    }
  }
  return best | (neg << sign_shift);
}

int oracle_encode_e4m3(double x) { return encode_nearest(x, 126, 7, oracle_e4m3_value); }
int oracle_encode_e2m1(double x) { return encode_nearest(x, 7, 3, oracle_e2m1_value); }

/* Quantise-and-write of cache rows.  Row i of src (dim fp32 values) goes to
 * row dst_row[i] of the destination (skipped when negative; past `rows` it is
 * skipped and RANGE_ROW is set).  A group holding a NaN or an infinity is
 * written as zero codes with the neutral scale and sets NONFINITE.
 *   format 1, FP8 block-32: s = amax / 448 (fp32; 1 when that is 0), codes
 *     E4M3(x / s); codes [rows, dim], scales fp32 [rows, dim/32].
 *   format 2, FP4 main KV: sc = E4M3(amax / 6), s = value(sc), codes
 *     E2M1(x / s) (0 when s is 0); codes [rows, dim/2], sf [rows, dim/16].
 *   format 3, MXFP4: s = 2^(floor(log2 amax) - 2) (1 when amax is 0), codes
 *     E2M1(x / s); codes [rows, dim/2], scales fp32 [rows, dim/32]; a scale
 *     outside [2^-23, 2^12] sets SCALE (0 as a scale: written as a zero group).
 * Element 2i of an E2M1 row sits in the low nibble of byte i. */
int oracle_encode_rows(int format, int64_t n, const float *src, int dim, const int64_t *dst_row,
                       uint8_t *codes, void *scales, int64_t rows) {
  int err = 0;
  const int gs = format == 2 ? 16 : 32;
  for (int64_t i = 0; i < n; ++i) {
    const int64_t r = dst_row[i];
    if (r < 0) continue;
    if (r >= rows) {
      err |= OR_ERR_RANGE_ROW;
      continue;
    }
    const float *x = src + i * dim;
    for (int g = 0; g < dim / gs; ++g) {
      float amax = 0.0f;
      int bad = 0;
      for (int e = 0; e < gs; ++e) {
        const float v = x[g * gs + e];
        if (!isfinite(v)) bad = 1;
        else if (fabsf(v) > amax) amax = fabsf(v);
      }
      float s = 1.0f;
      int zero = bad;
      uint8_t sf = 0;
      if (bad) {
        err |= OR_ERR_NONFINITE;
      } else if (format == 1) {
        s = amax / 448.0f;
        if (s == 0.0f) s = 1.0f;
      } else if (format == 2) {
        sf = (uint8_t)oracle_encode_e4m3((double)(amax / 6.0f));
        s = (float)oracle_e4m3_value(sf);
        if (s == 0.0f) zero = 1;
      } else if (amax > 0.0f) {
        int ex = 0;
        (void)frexpf(amax, &ex);
        s = ldexpf(1.0f, ex - 3);
        if (s == 0.0f || s < 0x1p-23f || s > 0x1p12f) err |= OR_ERR_SCALE;
        if (s == 0.0f) {
          s = 1.0f;
          zero = 1;
        }
      }
      for (int e = 0; e < gs; ++e) {
        const int d = g * gs + e;
        const float q = zero ? 0.0f : x[d] / s;
        if (format == 1) {
          codes[r * dim + d] = (uint8_t)oracle_encode_e4m3((double)q);
        } else {
          const int c = oracle_encode_e2m1((double)q);
          uint8_t *b = codes + r * (dim / 2) + d / 2;
          *b = (d & 1) ? (uint8_t)((*b & 0x0f) | (c << 4)) : (uint8_t)((*b & 0xf0) | c);
        }
      }
      if (format == 2) ((uint8_t *)scales)[r * (dim / 16) + g] = bad ? 0 : sf;
      else ((float *)scales)[r * (dim / 32) + g] = s;
    }
  }
  return err;
}

/* One MXFP4 row of `dim` elements decoded to double (used by the pins: the
 * index score's dot products cannot see the nibble order, which both operands
 * share, but the rows a quantiser writes must decode in this order). */
void oracle_decode_mxfp4_row(const uint8_t *codes, const float *scales, int dim, double *out) {
  for (int d = 0; d < dim; ++d) out[d] = mxfp4_elem(codes, scales, d);
}

/* One FP4 main-KV row of `dim` elements decoded to double (used by the pins). */
void oracle_decode_fp4kv_row(const uint8_t *codes, const uint8_t *sf, int dim,
                             double *out) {
  for (int d = 0; d < dim; ++d) out[d] = fp4kv_elem(codes, sf, d);
}

/* bf16 -> double (exact) and double -> bf16 with round-to-nearest-even. */
static double bf16_to_double(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* Index keys projected from the compressed main KV, written as MXFP4 cache
 * rows ("DeepSeek V4.1 Flash 建模", CSA2 card, compressor paragraph: index K is
 * projected from the compressed main KV; SGLang/Miles day-0 article sec. 5:
 * projection weights in BF16 with FP32 accumulation).  For source row i
 * (x: dim_in bf16 values) and output channel o (w row o: dim_in bf16 values):
 *   y[i][o] = sum_d x[i][d] * w[o][d]
 * formed in double (every bf16 x bf16 product is exact there, and so is the
 * sum while the products span fewer than about 37 binades) and rounded once
 * to fp32: the value an fp32 accumulation approximates.  The rows y[i] are
 * then encoded exactly as oracle_encode_rows format 3 (MXFP4) encodes rows,
 * into row dst_row[i] of (codes, scales).  y_out ([n, dim_out] fp32) receives
 * the unquantised rows when not NULL. */
int oracle_index_k_project(int64_t n, const uint16_t *x_bf16, int dim_in,
                           const uint16_t *w_bf16, int dim_out, const int64_t *dst_row,
                           uint8_t *codes, float *scales, int64_t rows, float *y_out) {
  float *y = (float *)malloc(sizeof(float) * (size_t)(n > 0 ? n : 1) * (size_t)dim_out);
  for (int64_t i = 0; i < n; ++i) {
    for (int o = 0; o < dim_out; ++o) {
      double acc = 0.0;
      for (int d = 0; d < dim_in; ++d)
        acc += bf16_to_double(x_bf16[i * dim_in + d]) * bf16_to_double(w_bf16[(int64_t)o * dim_in + d]);
      y[i * dim_out + o] = (float)acc;
    }
  }
  if (y_out) memcpy(y_out, y, sizeof(float) * (size_t)n * (size_t)dim_out);
  const int err = oracle_encode_rows(3, n, y, dim_out, dst_row, codes, scales, rows);
  free(y);
  return err;
}

uint16_t oracle_double_to_bf16(double x) {
  float f = (float)x; /* double -> float is itself RNE; then float -> bf16 RNE */
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7f800000u) == 0x7f800000u) { /* inf / nan pass through */
    uint16_t h = (uint16_t)(u >> 16);
    if (u & 0x007fffffu) h |= 0x40; /* keep NaN quiet */
    return h;
  }
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7fffu + lsb;
  return (uint16_t)(u >> 16);
}

/* ------------------------------------------------------------------------ */
/* Visibility over compressed positions                                       */
/* ------------------------------------------------------------------------ */

/* Number of compressed entries visible to the query at absolute position t
 * when each entry compresses m consecutive tokens without overlap. */
int64_t oracle_n_visible(int64_t t, int m) {
  if (t < 0) return 0;
  return (t + 1) / m;
}

/* ------------------------------------------------------------------------ */
/* a1: decoder bounded-replay tail layout                                     */
/* ------------------------------------------------------------------------ */

/* Per request r with extend length E_r and total length S_r after the extend:
 * T_r = min(W, E_r); the kept rows are the last T_r rows of this extend (rows
 * cu_E[r] + E_r - T_r ... of the packed extend), their absolute positions are
 * S_r - T_r ... S_r - 1 (never renumbered), and every kept row carries the
 * window lower bound S_r - T_r.  Returns the OR of data-error bits. */
int oracle_tail_layout(int32_t num_req, const int32_t *extend_len,
                       const int64_t *seq_len, int32_t window,
                       int32_t *tail_len, int32_t *cu_tail, int32_t *src_row,
                       int64_t *pos, int64_t *win_lo, int32_t *row_req,
                       int64_t capacity) {
  int err = 0;
  int64_t cu_e = 0, cu_t = 0;
  cu_tail[0] = 0;
  for (int r = 0; r < num_req; ++r) {
    int64_t e = extend_len[r], s = seq_len[r];
    int64_t t = 0;
    if (e < 0 || s < e) {
      err |= OR_ERR_BAD_EXTEND;
    } else {
      t = e < window ? e : window;
    }
    tail_len[r] = (int32_t)t;
    for (int64_t k = 0; k < t; ++k) {
      int64_t row = cu_t + k;
      if (row >= capacity) {
        err |= OR_ERR_CAPACITY;
        continue;
      }
      src_row[row] = (int32_t)(cu_e + e - t + k);
      pos[row] = s - t + k;
      win_lo[row] = s - t;
      if (row_req) row_req[row] = r;
    }
    if (e > 0) cu_e += e;
    cu_t += t;
    cu_tail[r + 1] = (int32_t)cu_t;
  }
  return err;
}

/* ------------------------------------------------------------------------ */
/* encoder-side bounded replay layout                                         */
/* ------------------------------------------------------------------------ */

/* Per request r with P_r cached prefix tokens (global entries and index keys
 * cached, SWA state gone) and E_r new tokens: the replayed part is the last
 * Rp_r = min(W, P_r) cached tokens, so the rows processed are the positions
 * P_r - Rp_r ... P_r + E_r - 1 in order.  A replayed row has no row in the
 * packed new-token input (src_row = -1); new row k - Rp_r of the request sits
 * at cu_E[r] + k - Rp_r.  Every row carries the window lower bound P_r - Rp_r
 * (local attention is cut where the rebuild starts).  Global entries: with m
 * tokens per entry, entry j is complete once token m*j + m - 1 exists, so the
 * cache already holds entries j < floor(P_r / m) and this extend completes
 * entries floor(P_r / m) <= j < floor((P_r + E_r) / m): entry_range[2r] and
 * entry_range[2r+1].  Returns the OR of data-error bits. */
int oracle_encoder_replay_layout(int32_t num_req, const int64_t *prefix_len,
                                 const int32_t *extend_len, int32_t window, int32_t ratio,
                                 int32_t *replay_len, int32_t *cu_rows, int32_t *src_row,
                                 int64_t *pos, int64_t *win_lo, int32_t *row_req,
                                 int64_t *entry_range, int64_t capacity) {
  int err = 0;
  int64_t cu_e = 0, cu_n = 0;
  cu_rows[0] = 0;
  for (int r = 0; r < num_req; ++r) {
    int64_t p = prefix_len[r], e = extend_len[r];
    int64_t rp = 0, n = 0;
    if (p < 0 || e < 0) {
      err |= OR_ERR_BAD_EXTEND;
      p = 0;
      e = 0;
    } else {
      rp = p < window ? p : window;
      n = rp + e;
    }
    replay_len[r] = (int32_t)rp;
    if (entry_range) {
      entry_range[2 * r] = p / ratio;
      entry_range[2 * r + 1] = (p + e) / ratio;
    }
    for (int64_t k = 0; k < n; ++k) {
      int64_t row = cu_n + k;
      if (row >= capacity) {
        err |= OR_ERR_CAPACITY;
        continue;
      }
      pos[row] = p - rp + k;
      win_lo[row] = p - rp;
      src_row[row] = k < rp ? -1 : (int32_t)(cu_e + (k - rp));
      if (row_req) row_req[row] = r;
    }
    cu_e += e;
    cu_n += n;
    cu_rows[r + 1] = (int32_t)cu_n;
  }
  return err;
}

/* ------------------------------------------------------------------------ */
/* row cut (gather) and scatter-back                                          */
/* ------------------------------------------------------------------------ */

/* dst row i = src row row_idx[i] for i < n (rows of row_bytes bytes).  A
 * negative index leaves dst row i as it was; an index >= src_rows does too and
 * sets the RANGE_ROW bit. */
int oracle_rows_gather(int64_t n, const int32_t *row_idx, const uint8_t *src, int64_t src_rows,
                       uint8_t *dst, int64_t row_bytes) {
  int err = 0;
  for (int64_t i = 0; i < n; ++i) {
    int64_t j = row_idx[i];
    if (j < 0) continue;
    if (j >= src_rows) {
      err |= OR_ERR_RANGE_ROW;
      continue;
    }
    memcpy(dst + i * row_bytes, src + j * row_bytes, (size_t)row_bytes);
  }
  return err;
}

/* dst row row_idx[i] = src row i for i < n; the dst rows no index names are
 * left as they were.  Negative indices are skipped; indices >= dst_rows are
 * skipped and set the RANGE_ROW bit. */
int oracle_rows_scatter(int64_t n, const int32_t *row_idx, const uint8_t *src, uint8_t *dst,
                        int64_t dst_rows, int64_t row_bytes) {
  int err = 0;
  for (int64_t i = 0; i < n; ++i) {
    int64_t j = row_idx[i];
    if (j < 0) continue;
    if (j >= dst_rows) {
      err |= OR_ERR_RANGE_ROW;
      continue;
    }
    memcpy(dst + j * row_bytes, src + i * row_bytes, (size_t)row_bytes);
  }
  return err;
}

/* ------------------------------------------------------------------------ */
/* a2-a4, a7: index scores                                                     */
/* ------------------------------------------------------------------------ */

/* Number of leading (non-negative) block ids in a candidate row. */
static int count_blocks(const int32_t *blocks, int max_blocks) {
  int n = 0;
  while (n < max_blocks && blocks[n] >= 0) ++n;
  return n;
}

/* s(q,j) = sum_h w[q,h] * max(0, sum_d Qi[q,h,d] * Ki[j,d]).
 * Full mode (cand_blocks == NULL): row q holds entries j = 0 .. n_vis-1.
 * Pool mode: row q holds slots s = 0 .. nb*block-1 of its candidate blocks;
 * slot s is entry blocks[q, s/block]*block + s%block, scored if visible and
 * -inf otherwise.  Columns past the row length are not written.  Scores are
 * produced in double and stored as the nearest float. */
int oracle_index_score(const oracle_batch *b, int n_heads, int head_dim,
                       const uint8_t *q_fp4, const float *q_scale,
                       const float *head_w, const uint8_t *k_fp4,
                       const float *k_scale, const int32_t *cand_blocks,
                       int block, int max_blocks, float *scores, int64_t ld) {
  int err = 0;
  const int qbytes = head_dim / 2, qgroups = head_dim / 32;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : err)
  for (int q = 0; q < b->num_q; ++q) {
    int r = b->q_req[q];
    int64_t n_vis = oracle_n_visible(b->q_pos[q], b->ratio);
    if (n_vis > b->kv_len[r]) {
      err |= OR_ERR_RANGE_CTX;
      n_vis = b->kv_len[r];
    }
    double *qv = (double *)malloc(sizeof(double) * n_heads * head_dim);
    double *kv = (double *)malloc(sizeof(double) * head_dim);
    for (int h = 0; h < n_heads; ++h)
      for (int d = 0; d < head_dim; ++d)
        qv[h * head_dim + d] =
            mxfp4_elem(q_fp4 + ((int64_t)q * n_heads + h) * qbytes,
                       q_scale + ((int64_t)q * n_heads + h) * qgroups, d);
    int64_t row_len;
    int nb = 0;
    if (cand_blocks) {
      nb = count_blocks(cand_blocks + (int64_t)q * max_blocks, max_blocks);
      row_len = (int64_t)nb * block;
    } else {
      row_len = n_vis;
    }
    if (row_len > ld) {
      err |= OR_ERR_LD;
      row_len = ld;
    }
    for (int64_t s = 0; s < row_len; ++s) {
      int64_t j = s;
      if (cand_blocks) {
        int64_t blk = cand_blocks[(int64_t)q * max_blocks + s / block];
        j = blk * block + s % block;
        if (j >= n_vis) {
          scores[(int64_t)q * ld + s] = -INFINITY;
          continue;
        }
      }
      int64_t row = b->kv_start[r] + j;
      for (int d = 0; d < head_dim; ++d)
        kv[d] = mxfp4_elem(k_fp4 + row * qbytes, k_scale + row * qgroups, d);
      double acc = 0.0;
      for (int h = 0; h < n_heads; ++h) {
        double dot = 0.0;
        for (int d = 0; d < head_dim; ++d) dot += qv[h * head_dim + d] * kv[d];
        double w = head_w ? (double)head_w[(int64_t)q * n_heads + h] : 1.0;
        acc += w * (dot > 0.0 ? dot : 0.0);
      }
      scores[(int64_t)q * ld + s] = (float)acc;
    }
    free(qv);
    free(kv);
  }
  return err;
}

/* ------------------------------------------------------------------------ */
/* a5, a7: top-K selection                                                    */
/* ------------------------------------------------------------------------ */

typedef struct {
  float s;
  int64_t j; /* entry id (tie-break key) */
} cand_t;

/* Pinned total order: score descending, then entry id ascending. */
static int cand_cmp(const void *a, const void *b) {
  const cand_t *x = (const cand_t *)a, *y = (const cand_t *)b;
  if (x->s > y->s) return -1;
  if (x->s < y->s) return 1;
  return (x->j > y->j) - (x->j < y->j);
}

/* Per query, the k entries with the highest scores among the visible entries
 * (full mode) or among the visible pool slots (pool mode), by the total order
 * above.  NaN and -inf scores are never selected; fewer than k eligible
 * entries leave -1 padding.  The result is a set: it is written sorted by
 * that order. */
int oracle_topk(const oracle_batch *b, const float *scores, int64_t ld, int k,
                const int32_t *cand_blocks, int block, int max_blocks,
                int32_t *idx, int32_t *count) {
  int err = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : err)
  for (int q = 0; q < b->num_q; ++q) {
    int r = b->q_req[q];
    int64_t n_vis = oracle_n_visible(b->q_pos[q], b->ratio);
    if (n_vis > b->kv_len[r]) {
      err |= OR_ERR_RANGE_CTX;
      n_vis = b->kv_len[r];
    }
    int64_t row_len;
    if (cand_blocks)
      row_len = (int64_t)count_blocks(cand_blocks + (int64_t)q * max_blocks,
                                      max_blocks) * block;
    else
      row_len = n_vis;
    if (row_len > ld) {
      err |= OR_ERR_LD;
      row_len = ld;
    }
    cand_t *c = (cand_t *)malloc(sizeof(cand_t) * (row_len > 0 ? row_len : 1));
    int64_t n = 0;
    for (int64_t s = 0; s < row_len; ++s) {
      int64_t j = s;
      if (cand_blocks) {
        j = (int64_t)cand_blocks[(int64_t)q * max_blocks + s / block] * block +
            s % block;
        if (j >= n_vis) continue;
      }
      float v = scores[(int64_t)q * ld + s];
      if (isnan(v) || v == -INFINITY) continue;
      c[n].s = v;
      c[n].j = j;
      ++n;
    }
    qsort(c, (size_t)n, sizeof(cand_t), cand_cmp);
    int take = n < k ? (int)n : k;
    for (int i = 0; i < k; ++i)
      idx[(int64_t)q * k + i] = i < take ? (int32_t)c[i].j : -1;
    count[q] = take;
    free(c);
  }
  return err;
}

/* ------------------------------------------------------------------------ */
/* a6: hierarchical candidate blocks                                          */
/* ------------------------------------------------------------------------ */

typedef struct {
  float s;
  int64_t b;
} blk_t;

static int blk_cmp(const void *a, const void *bb) {
  const blk_t *x = (const blk_t *)a, *y = (const blk_t *)bb;
  if (x->s > y->s) return -1;
  if (x->s < y->s) return 1;
  return (x->b > y->b) - (x->b < y->b);
}

static int i64_cmp(const void *a, const void *b) {
  int64_t x = *(const int64_t *)a, y = *(const int64_t *)b;
  return (x > y) - (x < y);
}

/* Blocks are aligned groups of `block` consecutive entries.  The block score
 * is the maximum score over the block's visible entries (NaN ignored; -inf if
 * none).  With B = ceil(n_vis/block) blocks: B <= max_blocks keeps all of
 * them; otherwise the latest block B-1 takes one slot and the remaining
 * max_blocks-1 slots go to the best blocks among 0..B-2 by (block score desc,
 * block id asc).  The pool is a position budget, so it is always filled to
 * min(B, max_blocks) blocks whatever their scores.  Output ascending, -1
 * padded.  The query's own top-k over entries is written too (oracle_topk). */
int oracle_topk_candidates(const oracle_batch *b, const float *scores,
                           int64_t ld, int k, int block, int max_blocks,
                           int32_t *idx, int32_t *count, int32_t *blocks,
                           int32_t *nblocks) {
  int err = oracle_topk(b, scores, ld, k, NULL, block, max_blocks, idx, count);
#pragma omp parallel for schedule(dynamic, 1) reduction(| : err)
  for (int q = 0; q < b->num_q; ++q) {
    int r = b->q_req[q];
    int64_t n_vis = oracle_n_visible(b->q_pos[q], b->ratio);
    if (n_vis > b->kv_len[r]) n_vis = b->kv_len[r];
    if (n_vis > ld) n_vis = ld;
    int64_t nb_all = (n_vis + block - 1) / block;
    int32_t *out = blocks + (int64_t)q * max_blocks;
    int64_t keep = 0;
    int64_t *chosen = (int64_t *)malloc(sizeof(int64_t) * (max_blocks + 1));
    if (nb_all <= max_blocks) {
      for (int64_t bb = 0; bb < nb_all; ++bb) chosen[keep++] = bb;
    } else {
      blk_t *bs = (blk_t *)malloc(sizeof(blk_t) * nb_all);
      for (int64_t bb = 0; bb < nb_all - 1; ++bb) {
        float m = -INFINITY;
        for (int64_t j = bb * block; j < (bb + 1) * block && j < n_vis; ++j) {
          float v = scores[(int64_t)q * ld + j];
          if (!isnan(v) && v > m) m = v;
        }
        bs[bb].s = m;
        bs[bb].b = bb;
      }
      qsort(bs, (size_t)(nb_all - 1), sizeof(blk_t), blk_cmp);
      for (int i = 0; i < max_blocks - 1; ++i) chosen[keep++] = bs[i].b;
      chosen[keep++] = nb_all - 1; /* the block holding the latest position */
      free(bs);
      qsort(chosen, (size_t)keep, sizeof(int64_t), i64_cmp);
    }
    for (int i = 0; i < max_blocks; ++i) out[i] = i < keep ? (int32_t)chosen[i] : -1;
    nblocks[q] = (int32_t)keep;
    free(chosen);
  }
  return err;
}

/* ------------------------------------------------------------------------ */
/* a8-a10: sparse + sliding-window attention under one softmax                */
/* ------------------------------------------------------------------------ */

/* For query q (request r, absolute position t) and head h:
 *   rows = { KV[kv_start[r]+j] : j in idx[q], j >= 0 }            (selected)
 *        u { SWA row of position p : lo <= p <= t }                 (window)
 *   lo   = max(win_lo[q], t - window + 1, 0)
 *   l_i  = sm_scale * <Q[q,h], row_i>      (the row is key and value)
 *   O    = sum_i e^{l_i} row_i / (sum_i e^{l_i} + e^{sink_h})
 *   lse  = log(sum_i e^{l_i} + e^{sink_h})
 * evaluated as a two-pass softmax in double.  The union is not de-duplicated.
 * Selected ids outside [0, n_vis) or past kv_len are skipped (error bit 1);
 * window positions without a stored SWA row are skipped (error bit 2).  A
 * query with no rows and no sink gets O = 0 and lse = -inf.  O is rounded to
 * bf16 (RNE), lse stored as float. */
/* Selected rows come from the main KV pool in one of two formats: FP8 block-32
 * (kv_codes [Nkv, dim] E4M3 + kv_scales fp32 [Nkv, dim/32]) or FP4
 * (kv_codes [Nkv, dim/2] E2M1 + kv_sf E4M3 [Nkv, dim/16]).  Window rows are
 * always FP8 block-32 (mixed-precision card: SWA stays FP8). */
static int attn_core(const oracle_batch *b, int n_heads, int dim, const uint16_t *q_bf16,
                     int kv_fp4, const uint8_t *kv_codes, const float *kv_scale,
                     const uint8_t *kv_sf, const int32_t *idx, int k, const uint8_t *swa_fp8,
                     const float *swa_scale, const int64_t *win_lo, int window,
                     double sm_scale, const float *sink, uint16_t *out_bf16, float *lse) {
  int err = 0;
  const int nsc = dim / 32;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : err)
  for (int q = 0; q < b->num_q; ++q) {
    int r = b->q_req[q];
    int64_t t = b->q_pos[q];
    int64_t n_vis = oracle_n_visible(t, b->ratio);
    int cap = k + window;
    double *rows = (double *)malloc(sizeof(double) * (size_t)cap * dim);
    int nrows = 0;
    /* selected compressed rows */
    for (int i = 0; i < k && idx; ++i) {
      int64_t j = idx[(int64_t)q * k + i];
      if (j < 0) continue;
      if (j >= n_vis || j >= b->kv_len[r]) {
        err |= OR_ERR_RANGE_IDX;
        continue;
      }
      int64_t row = b->kv_start[r] + j;
      for (int d = 0; d < dim; ++d)
        rows[(size_t)nrows * dim + d] =
            kv_fp4 ? fp4kv_elem(kv_codes + row * (dim / 2), kv_sf + row * (dim / 16), d)
                   : fp8_elem(kv_codes + row * dim, kv_scale + row * nsc, d);
      ++nrows;
    }
    /* the query's own sliding window */
    int64_t lo = t - window + 1;
    if (win_lo && win_lo[q] > lo) lo = win_lo[q];
    if (lo < 0) lo = 0;
    for (int64_t p = lo; p <= t; ++p) {
      int64_t off = p - b->swa_pos0[r];
      if (off < 0 || off >= b->swa_len[r]) {
        err |= OR_ERR_RANGE_WINDOW;
        continue;
      }
      int64_t row = b->swa_start[r] + off;
      for (int d = 0; d < dim; ++d)
        rows[(size_t)nrows * dim + d] =
            fp8_elem(swa_fp8 + row * dim, swa_scale + row * nsc, d);
      ++nrows;
    }
    double *logit = (double *)malloc(sizeof(double) * (nrows > 0 ? nrows : 1));
    double *o = (double *)malloc(sizeof(double) * dim);
    for (int h = 0; h < n_heads; ++h) {
      const uint16_t *qh = q_bf16 + ((int64_t)q * n_heads + h) * dim;
      double m = -INFINITY;
      for (int i = 0; i < nrows; ++i) {
        double dot = 0.0;
        for (int d = 0; d < dim; ++d)
          dot += bf16_to_double(qh[d]) * rows[(size_t)i * dim + d];
        logit[i] = sm_scale * dot;
        if (logit[i] > m) m = logit[i];
      }
      double sk = sink ? (double)sink[h] : -INFINITY;
      if (sk > m) m = sk;
      double denom = 0.0;
      for (int d = 0; d < dim; ++d) o[d] = 0.0;
      if (m != -INFINITY) {
        for (int i = 0; i < nrows; ++i) {
          double p = exp(logit[i] - m);
          denom += p;
          for (int d = 0; d < dim; ++d) o[d] += p * rows[(size_t)i * dim + d];
        }
        if (sink) denom += exp(sk - m);
      }
      uint16_t *oh = out_bf16 + ((int64_t)q * n_heads + h) * dim;
      for (int d = 0; d < dim; ++d)
        oh[d] = oracle_double_to_bf16(denom > 0.0 ? o[d] / denom : 0.0);
      if (lse)
        lse[(int64_t)q * n_heads + h] =
            denom > 0.0 ? (float)(m + log(denom)) : -INFINITY;
    }
    free(rows);
    free(logit);
    free(o);
  }
  return err;
}

int oracle_sparse_swa_attn(const oracle_batch *b, int n_heads, int dim,
                           const uint16_t *q_bf16, const uint8_t *kv_fp8,
                           const float *kv_scale, const int32_t *idx, int k,
                           const uint8_t *swa_fp8, const float *swa_scale,
                           const int64_t *win_lo, int window, double sm_scale,
                           const float *sink, uint16_t *out_bf16, float *lse) {
  return attn_core(b, n_heads, dim, q_bf16, 0, kv_fp8, kv_scale, NULL, idx, k, swa_fp8,
                   swa_scale, win_lo, window, sm_scale, sink, out_bf16, lse);
}

/* The same attention with the selected rows read from the FP4 main-KV pool. */
int oracle_sparse_swa_attn_fp4kv(const oracle_batch *b, int n_heads, int dim,
                                 const uint16_t *q_bf16, const uint8_t *kv_fp4,
                                 const uint8_t *kv_sf, const int32_t *idx, int k,
                                 const uint8_t *swa_fp8, const float *swa_scale,
                                 const int64_t *win_lo, int window, double sm_scale,
                                 const float *sink, uint16_t *out_bf16, float *lse) {
  return attn_core(b, n_heads, dim, q_bf16, 1, kv_fp4, NULL, kv_sf, idx, k, swa_fp8,
                   swa_scale, win_lo, window, sm_scale, sink, out_bf16, lse);
}
