/*
 * CPU oracle for split-tier paged decode attention (test infrastructure only).
 *
 * A plain, slow, double-precision statement of what the hot path computes, used
 * to check the CUDA library.  It shares no code, header or constant with the
 * CUDA path; only the seeded input generator is common to both.  Nothing in the
 * product path may call it.
 *
 * Sources (web pages about ActiveKV, by their titles):
 *   [FMT]   "model quantization", section "An 8-bit page format shaped for its
 *           kernel": key scale per channel = sqrt of the channel's RMS over the
 *           page, normalised so the channel scales multiply to one, clamped to
 *           2^+-14; a per-token-and-head factor covers the rest; symmetric codes
 *           in -127..127; values carry one scale per channel per page.
 *   [ATT]   "SYCL", section "Attention that reads 8-bit history": the separable
 *           key scale (per-token factor applied after the dot), PV on raw codes
 *           rescaled per page.  The method is an exact re-association of
 *           "dequantise, then attend", so this oracle dequantises and attends.
 *   [MERGE] "SYCL", section "A merge that joins the tiers": partials (output plus
 *           log-sum-exp) folded into one accumulator; -inf is a valid empty partial.
 *   [TIERS] "ActiveKV", section "The idea": recent context exact, older history
 *           8-bit, joined with exact attention arithmetic.
 *   [LOSSLESS] "model quantization", section "A lossless tier first": 13 bits per
 *           value (an 18.7 % saving) with a raw fallback when a plane needs more
 *           than a 32-entry table.
 *   [IQ]    "SYCL", section "Attention that reads 8-bit history": the kernel keeps
 *           an integer query cache of 8 rows x 256 channels (2 KB) and a
 *           two-by-two experiment decided which products run on integers.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   - scales are stored as float32; key channel scales are rounded to float32 by
 *     compensated rounding so that their product stays 1;
 *   - normalisation is by the geometric mean, applied before the clamp; a channel
 *     with zero RMS takes a = 2^-63 before the logarithm;
 *   - per-token key factor r_t = max_c |k_tc / s_c| / 127, value scale
 *     u_c = max_t |v_tc| / 127 (absmax), both in float32;
 *   - codes: two correctly rounded float32 divisions (k / s_c, then / r_t),
 *     rint (half to even), clamp to +-127; a zero scale gives zero codes;
 *   - softmax scale 1/sqrt(d), log-sum-exp in natural-log units; an empty range
 *     gives o = 0, lse = -inf;
 *   - lossless tier: a plane is one page-head's keys (or values); the 32-entry
 *     table holds the plane's distinct BF16 exponent fields, so a value is its
 *     sign and mantissa (8 bits) plus a 5-bit table index;
 *   - integer query (the variant with integer QK products): the query folded with
 *     the page's key channel scales, q'_c = q_c s_c, is coded per page and query
 *     row with the absmax rule of the key codes: m = max_c |q'_c|, alpha = m / 127,
 *     qi_c = rint(q'_c * (127 / m)) clamped to +-127, every step in float32 (one
 *     division for 127 / m, one for m / 127, then products); m = 0 gives alpha = 0
 *     and zero codes.  The scores are alpha * r_t * sum_c qi_c kc_tc.
 *
 * Record layout of one 8-bit page-head (35,072 bytes):
 *   u8    kc[64][256]      keys, token-major       offset 0
 *   u8    vc[256][64]      values, channel-major   offset 16384
 *   f32   ks_chan[256]     key channel scale s_c   offset 32768
 *   f32   ks_tok[64]       key token factor r_t    offset 33792
 *   f32   vs_chan[256]     value channel scale u_c offset 34048
 * with three position swizzles (the format is shaped for the kernel that reads it):
 *   key code (t, c)   at byte t*256 + (c XOR 64 * (t mod 2))
 *   value code (c, t) at byte c*64 + (t XOR 32 * ((c / 2) mod 2))
 *   s_c               at float (c XOR 8 * ((c / 32) mod 2))
 * and each code c in [-127, 127] stored as the byte c + 128 (offset binary).
 * Dequantised: k_tc = kc_tc * s_c * r_t,  v_tc = vc_tc * u_c.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define T_PAGE 64
#define D_HEAD 256
#define REC_BYTES 35072
#define OFF_KC 0
#define OFF_VC 16384
#define OFF_KS_CHAN 32768
#define OFF_KS_TOK 33792
#define OFF_VS_CHAN 34048

/* positions inside a record (see the layout above) */
static int kc_pos(int t, int c) { return t * D_HEAD + (c ^ (64 * (t & 1))); }
static int vc_pos(int c, int t) { return c * T_PAGE + (t ^ (32 * ((c >> 1) & 1))); }
static int ks_pos(int c) { return c ^ (8 * ((c >> 5) & 1)); }

static double bf16_value(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

static float bf16_float(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* ================================================================ quantiser */

/*
 * Compensated rounding of the key channel scales (the reading that makes the
 * stored float32 scales multiply to one [FMT]): channel c may be stored as its
 * lower or its upper float32 neighbour, whose log errors ln(neighbour / shat_c)
 * are dlo[c] <= 0 <= dhi[c].  Walk c = 0 .. n-1 keeping the running log error E
 * of the product (E = 0 at the start); channel c takes the lower neighbour when
 * |E + dlo[c]| <= |E + dhi[c]| (so the lower one on a tie), else the upper one,
 * and E grows by the chosen error.  take_hi[c] = 1 marks the upper neighbour.
 */
void orc_compensated_walk(int n, const double* dlo, const double* dhi, int* take_hi) {
  double E = 0.0;
  for (int c = 0; c < n; ++c) {
    if (fabs(E + dlo[c]) <= fabs(E + dhi[c])) {
      take_hi[c] = 0;
      E += dlo[c];
    } else {
      take_hi[c] = 1;
      E += dhi[c];
    }
  }
}

/*
 * Key channel scales of one page-head [FMT].
 *   ms_c  = mean_t k_tc^2 (double);  a_c = sqrt(sqrt(ms_c))   (sqrt of the RMS)
 *   g     = exp(mean_c ln a_c)       (geometric mean, so prod_c a_c/g = 1)
 *   shat_c= clamp(a_c / g, 2^-14, 2^14)
 *   s_c   = a float32 neighbour of shat_c chosen by compensated rounding: walk the
 *           channels in order keeping E = sum (ln s - ln shat); take whichever
 *           neighbour leaves |E| smaller (the lower one on a tie).
 * Returns the number of channels the clamp engaged.
 */
int orc_channel_scales(const uint16_t* k, float* s_out, double* shat_out) {
  double a[D_HEAD], shat[D_HEAD];
  double sum_ln = 0.0;
  for (int c = 0; c < D_HEAD; ++c) {
    double ms = 0.0;
    for (int t = 0; t < T_PAGE; ++t) {
      double x = bf16_value(k[t * D_HEAD + c]);
      ms += x * x;
    }
    ms /= T_PAGE;
    double rms = sqrt(ms);
    a[c] = rms > 0.0 ? sqrt(rms) : ldexp(1.0, -63);
    sum_ln += log(a[c]);
  }
  double g = exp(sum_ln / D_HEAD);
  int clamped = 0;
  const double lo_b = ldexp(1.0, -14), hi_b = ldexp(1.0, 14);
  for (int c = 0; c < D_HEAD; ++c) {
    double v = a[c] / g;
    if (v < lo_b) { v = lo_b; ++clamped; }
    if (v > hi_b) { v = hi_b; ++clamped; }
    shat[c] = v;
  }
  /* the two float32 neighbours of each shat_c and their log errors; a channel
     whose shat_c is a float has lo = hi and zero errors (it leaves E unchanged) */
  float lo[D_HEAD], hi[D_HEAD];
  double dlo[D_HEAD], dhi[D_HEAD];
  for (int c = 0; c < D_HEAD; ++c) {
    double sh = shat[c];
    float f = (float)sh;
    if ((double)f == sh) {
      lo[c] = hi[c] = f;
      dlo[c] = dhi[c] = 0.0;
      continue;
    }
    lo[c] = ((double)f < sh) ? f : nextafterf(f, 0.0f);
    hi[c] = nextafterf(lo[c], INFINITY);
    dlo[c] = log((double)lo[c] / sh);
    dhi[c] = log((double)hi[c] / sh);
  }
  int take_hi[D_HEAD];
  orc_compensated_walk(D_HEAD, dlo, dhi, take_hi);
  for (int c = 0; c < D_HEAD; ++c) s_out[c] = take_hi[c] ? hi[c] : lo[c];
  if (shat_out)
    for (int c = 0; c < D_HEAD; ++c) shat_out[c] = shat[c];
  return clamped;
}

static int8_t code_of(float x, float scale) {
  if (!(scale > 0.0f)) return 0;
  float y = rintf(x / scale); /* float32 IEEE division, then half-to-even */
  if (y > 127.0f) y = 127.0f;
  if (y < -127.0f) y = -127.0f;
  return (int8_t)y;
}

/*
 * Codes of one page-head given all three scale arrays [FMT]:
 *   kc_tc = clamp(rint((k_tc / s_c) / r_t)),  vc_tc = clamp(rint(v_tc / u_c)).
 * The scales are copied into the record unchanged.
 */
void orc_codes_given(const uint16_t* k, const uint16_t* v, const float* ks_chan, const float* ks_tok,
                     const float* vs_chan, uint8_t* rec) {
  uint8_t* kc = rec + OFF_KC;
  uint8_t* vc = rec + OFF_VC;
  for (int t = 0; t < T_PAGE; ++t)
    for (int c = 0; c < D_HEAD; ++c) {
      float y = bf16_float(k[t * D_HEAD + c]) / ks_chan[c];
      kc[kc_pos(t, c)] = (uint8_t)(code_of(y, ks_tok[t]) + 128);
      vc[vc_pos(c, t)] = (uint8_t)(code_of(bf16_float(v[t * D_HEAD + c]), vs_chan[c]) + 128);
    }
  float* ks = (float*)(rec + OFF_KS_CHAN);
  for (int c = 0; c < D_HEAD; ++c) ks[ks_pos(c)] = ks_chan[c];
  memcpy(rec + OFF_KS_TOK, ks_tok, 4 * T_PAGE);
  memcpy(rec + OFF_VS_CHAN, vs_chan, 4 * D_HEAD);
}

/* Full conversion of one page-head [FMT]: scales, then codes.  Returns clamp count. */
int orc_quantize_page_head(const uint16_t* k, const uint16_t* v, uint8_t* rec) {
  float s[D_HEAD], r[T_PAGE], u[D_HEAD];
  int clamped = orc_channel_scales(k, s, 0);
  for (int t = 0; t < T_PAGE; ++t) {
    float m = 0.0f;
    for (int c = 0; c < D_HEAD; ++c) {
      float y = fabsf(bf16_float(k[t * D_HEAD + c]) / s[c]);
      if (y > m) m = y;
    }
    r[t] = m / 127.0f;
  }
  for (int c = 0; c < D_HEAD; ++c) {
    float m = 0.0f;
    for (int t = 0; t < T_PAGE; ++t) {
      float y = fabsf(bf16_float(v[t * D_HEAD + c]));
      if (y > m) m = y;
    }
    u[c] = m / 127.0f;
  }
  orc_codes_given(k, v, s, r, u, rec);
  return clamped;
}

/* Convert n_pages pages of a [slot][H][64][256] BF16 pool into records at
 * rec_pool + (dst_slot * H + h) * 35072. */
void orc_quantize_pages(int H, const uint16_t* k_pool, const uint16_t* v_pool, const int32_t* src_slots,
                        const int32_t* dst_slots, int n_pages, uint8_t* rec_pool) {
  const int64_t ph = (int64_t)T_PAGE * D_HEAD;
  for (int p = 0; p < n_pages; ++p)
    for (int h = 0; h < H; ++h) {
      int64_t src = ((int64_t)src_slots[p] * H + h) * ph;
      orc_quantize_page_head(k_pool + src, v_pool + src,
                             rec_pool + ((int64_t)dst_slots[p] * H + h) * REC_BYTES);
    }
}

/* ============================================================ lossless tier */

/*
 * Lossless 13-bit plane [LOSSLESS].  A plane is one page-head's keys (or values):
 * 64 x 256 BF16 values in token-major order.  Each BF16 value is a sign bit, an
 * 8-bit exponent field and a 7-bit mantissa.  When the plane holds at most 32
 * distinct exponent fields, each value is stored as its sign and mantissa (one
 * byte) plus the 5-bit position of its exponent in the plane's table of distinct
 * exponents (sorted ascending): 8 + 5 = 13 bits per value.  Otherwise the plane is
 * stored raw (16 bits per value).  Encoded plane, 26,656 bytes:
 *   u8 table[32]      distinct exponent fields, ascending; unused entries 0   offset 0
 *   u8 sm[16384]      (sign << 7) | mantissa of value i                     offset 32
 *   u8 lo4[8192]      index bits 0-3: value 2j in the low nibble of byte j,
 *                     value 2j + 1 in the high nibble                        offset 16416
 *   u8 hi1[2048]      index bit 4 of value 8j + b in bit b of byte j          offset 24608
 * Raw plane, 32,768 bytes: the BF16 values, little-endian.
 * Page-head record: u32 k_bytes, u32 v_bytes, u32 0, u32 0 (16 bytes), then the
 * key plane, then the value plane (k_bytes and v_bytes are 26656 or 32768).
 */
#define PLANE_VALUES (T_PAGE * D_HEAD)
#define PLANE_ENC_BYTES 26656
#define PLANE_RAW_BYTES 32768
#define P13_HEADER 16
#define P13_RECORD_BYTES (P13_HEADER + 2 * PLANE_RAW_BYTES)

/* Encode one plane into out; returns the bytes written. */
int orc_pack13_plane(const uint16_t* v, uint8_t* out) {
  int present[256] = {0};
  for (int i = 0; i < PLANE_VALUES; ++i) present[(v[i] >> 7) & 0xFF] = 1;
  uint8_t table[32];
  int n = 0;
  for (int e = 0; e < 256; ++e)
    if (present[e]) {
      if (n == 32) { /* a 33rd exponent: raw fallback */
        for (int i = 0; i < PLANE_VALUES; ++i) {
          out[2 * i] = (uint8_t)(v[i] & 0xFF);
          out[2 * i + 1] = (uint8_t)(v[i] >> 8);
        }
        return PLANE_RAW_BYTES;
      }
      table[n++] = (uint8_t)e;
    }
  memset(out, 0, PLANE_ENC_BYTES);
  for (int k = 0; k < n; ++k) out[k] = table[k];
  uint8_t* sm = out + 32;
  uint8_t* lo4 = out + 32 + 16384;
  uint8_t* hi1 = out + 32 + 16384 + 8192;
  for (int i = 0; i < PLANE_VALUES; ++i) {
    int e = (v[i] >> 7) & 0xFF;
    int idx = 0;
    while (table[idx] != e) ++idx; /* e is in the table */
    sm[i] = (uint8_t)(((v[i] >> 8) & 0x80) | (v[i] & 0x7F));
    lo4[i / 2] |= (uint8_t)((idx & 15) << (4 * (i % 2)));
    hi1[i / 8] |= (uint8_t)((idx >> 4) << (i % 8));
  }
  return PLANE_ENC_BYTES;
}

/* Decode a plane of nbytes (26656 or 32768) bytes; returns 0, or -1 for any other size. */
int orc_unpack13_plane(const uint8_t* in, int nbytes, uint16_t* v) {
  if (nbytes == PLANE_RAW_BYTES) {
    for (int i = 0; i < PLANE_VALUES; ++i) v[i] = (uint16_t)(in[2 * i] | (in[2 * i + 1] << 8));
    return 0;
  }
  if (nbytes != PLANE_ENC_BYTES) return -1;
  const uint8_t* sm = in + 32;
  const uint8_t* lo4 = in + 32 + 16384;
  const uint8_t* hi1 = in + 32 + 16384 + 8192;
  for (int i = 0; i < PLANE_VALUES; ++i) {
    int idx = ((lo4[i / 2] >> (4 * (i % 2))) & 15) | (((hi1[i / 8] >> (i % 8)) & 1) << 4);
    int e = in[idx];
    v[i] = (uint16_t)(((sm[i] & 0x80) << 8) | (e << 7) | (sm[i] & 0x7F));
  }
  return 0;
}

static void put_u32(uint8_t* p, uint32_t x) {
  for (int b = 0; b < 4; ++b) p[b] = (uint8_t)(x >> (8 * b));
}
static uint32_t get_u32(const uint8_t* p) {
  return (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) | ((uint32_t)p[3] << 24);
}

/* One page-head record (at most 65,552 bytes); returns its size. */
int orc_pack13_page_head(const uint16_t* k, const uint16_t* v, uint8_t* rec) {
  memset(rec, 0, P13_HEADER);
  int kb = orc_pack13_plane(k, rec + P13_HEADER);
  int vb = orc_pack13_plane(v, rec + P13_HEADER + kb);
  put_u32(rec, (uint32_t)kb);
  put_u32(rec + 4, (uint32_t)vb);
  return P13_HEADER + kb + vb;
}

/* Inverse of orc_pack13_page_head; returns 0, or -1 for a malformed header. */
int orc_unpack13_page_head(const uint8_t* rec, uint16_t* k, uint16_t* v) {
  int kb = (int)get_u32(rec), vb = (int)get_u32(rec + 4);
  if (orc_unpack13_plane(rec + P13_HEADER, kb, k) != 0) return -1;
  return orc_unpack13_plane(rec + P13_HEADER + kb, vb, v);
}

/* Pack n_pages pages of a [slot][H][64][256] BF16 pool into 65,552-byte slots of
 * pack_pool: page-head (src_slots[i], h) -> slot dst_slots[i] * H + h. */
void orc_pack13_pages(int H, const uint16_t* k_pool, const uint16_t* v_pool, const int32_t* src_slots,
                      const int32_t* dst_slots, int n_pages, uint8_t* pack_pool) {
  const int64_t ph = (int64_t)PLANE_VALUES;
  for (int p = 0; p < n_pages; ++p)
    for (int h = 0; h < H; ++h) {
      int64_t src = ((int64_t)src_slots[p] * H + h) * ph;
      uint8_t* rec = pack_pool + ((int64_t)dst_slots[p] * H + h) * P13_RECORD_BYTES;
      memset(rec, 0, P13_RECORD_BYTES);
      orc_pack13_page_head(k_pool + src, v_pool + src, rec);
    }
}

/* ================================================================ attention */

/*
 * Where the rows of one attention come from: a function that fills row[0..d)
 * with key (or value) i of the range, dequantised to double.
 */
typedef void (*row_fn)(const void* src, int i, double* row);

/*
 * Softmax of one query row over n precomputed scores s_t, in double:
 *   m = max_t s_t;  l = sum_t exp(s_t - m);  o = sum_t exp(s_t - m) v_t / l;
 *   lse = m + ln l.   n = 0 gives o = 0 and lse = -inf (the empty partial).
 * value_row(src, t, .) supplies v_t.
 */
static void attend_scores(int n, int d, const double* s, row_fn value_row, const void* src, double* orow,
                          double* lse) {
  for (int c = 0; c < d; ++c) orow[c] = 0.0;
  if (n == 0) {
    *lse = -INFINITY;
    return;
  }
  double m = -INFINITY;
  for (int t = 0; t < n; ++t)
    if (s[t] > m) m = s[t];
  double l = 0.0;
  double* v = (double*)malloc(sizeof(double) * d);
  for (int t = 0; t < n; ++t) {
    double w = exp(s[t] - m);
    l += w;
    value_row(src, t, v);
    for (int c = 0; c < d; ++c) orow[c] += w * v[c];
  }
  free(v);
  for (int c = 0; c < d; ++c) orow[c] /= l;
  *lse = m + log(l);
}

/*
 * Softmax attention of one query row over n tokens, in double:
 *   s_t = scale * q . k_t, then attend_scores.
 */
static void attend_row(int n, int d, const double* q, row_fn key_row, row_fn value_row, const void* src,
                       double scale, double* orow, double* lse) {
  double* s = (double*)malloc(sizeof(double) * (n > 0 ? n : 1));
  double* k = (double*)malloc(sizeof(double) * d);
  for (int t = 0; t < n; ++t) {
    key_row(src, t, k);
    double acc = 0.0;
    for (int c = 0; c < d; ++c) acc += q[c] * k[c];
    s[t] = scale * acc;
  }
  free(k);
  attend_scores(n, d, s, value_row, src, orow, lse);
  free(s);
}

/* dense [n][d] arrays of keys and values */
typedef struct {
  int d;
  const double *K, *V;
} dense_src;
static void dense_key(const void* p, int i, double* row) {
  const dense_src* S = (const dense_src*)p;
  memcpy(row, S->K + (int64_t)i * S->d, sizeof(double) * S->d);
}
static void dense_value(const void* p, int i, double* row) {
  const dense_src* S = (const dense_src*)p;
  memcpy(row, S->V + (int64_t)i * S->d, sizeof(double) * S->d);
}

/*
 * Softmax attention of `rows` query rows over n tokens (dense K, V), in double.
 */
void orc_attend(int n, int d, int rows, const double* q, const double* K, const double* V, double scale,
                double* o, double* lse) {
  dense_src S = {d, K, V};
  for (int r = 0; r < rows; ++r)
    attend_row(n, d, q + (int64_t)r * d, dense_key, dense_value, &S, scale, o + (int64_t)r * d, lse + r);
}

/* BF16 tokens [tok_begin, ...) of KV head h in a paged history: token t lives in
 * slot page_table[t / 64], row t % 64 [ATT, MERGE]. */
typedef struct {
  int H, h, tok_begin;
  const uint16_t *k_pool, *v_pool;
  const int32_t* page_table;
} exact_src;
static int64_t exact_base(const exact_src* S, int i) {
  int t = S->tok_begin + i;
  int64_t slot = S->page_table[t / T_PAGE];
  return ((slot * S->H + S->h) * T_PAGE + t % T_PAGE) * (int64_t)D_HEAD;
}
static void exact_key(const void* p, int i, double* row) {
  const exact_src* S = (const exact_src*)p;
  int64_t base = exact_base(S, i);
  for (int c = 0; c < D_HEAD; ++c) row[c] = bf16_value(S->k_pool[base + c]);
}
static void exact_value(const void* p, int i, double* row) {
  const exact_src* S = (const exact_src*)p;
  int64_t base = exact_base(S, i);
  for (int c = 0; c < D_HEAD; ++c) row[c] = bf16_value(S->v_pool[base + c]);
}

/* 8-bit pages [page_begin, ...) of KV head h, page p in slot page_table8[p],
 * dequantised [FMT]: k_tc = kc_tc s_c r_t, v_tc = vc_tc u_c. */
typedef struct {
  int H, h, page_begin;
  const uint8_t* rec_pool;
  const int32_t* page_table8;
} int8_src;
static const uint8_t* int8_record(const int8_src* S, int i) {
  return S->rec_pool + ((int64_t)S->page_table8[S->page_begin + i / T_PAGE] * S->H + S->h) * REC_BYTES;
}
static void int8_key(const void* p, int i, double* row) {
  const uint8_t* rec = int8_record((const int8_src*)p, i);
  const int t = i % T_PAGE;
  float s_stored[D_HEAD], r;
  memcpy(s_stored, rec + OFF_KS_CHAN, sizeof s_stored);
  memcpy(&r, rec + OFF_KS_TOK + 4 * t, 4);
  for (int c = 0; c < D_HEAD; ++c)
    row[c] = (double)((int)rec[OFF_KC + kc_pos(t, c)] - 128) * (double)s_stored[ks_pos(c)] * (double)r;
}
static void int8_value(const void* p, int i, double* row) {
  const uint8_t* rec = int8_record((const int8_src*)p, i);
  const int t = i % T_PAGE;
  float u[D_HEAD];
  memcpy(u, rec + OFF_VS_CHAN, sizeof u);
  for (int c = 0; c < D_HEAD; ++c) row[c] = (double)((int)rec[OFF_VC + vc_pos(c, t)] - 128) * (double)u[c];
}

static void query_row(const uint16_t* q, int r, double* qd) {
  for (int c = 0; c < D_HEAD; ++c) qd[c] = bf16_value(q[(int64_t)r * D_HEAD + c]);
}

/* Exact-tier partial of query row g of KV head h [ATT, MERGE] over BF16 tokens
 * [tok_begin, tok_end); q is [H*G][256], the result goes to row h*G + g. */
static void partial_exact_row(int H, int G, int h, int g, const uint16_t* q, const uint16_t* k_pool,
                              const uint16_t* v_pool, const int32_t* page_table, int tok_begin, int tok_end,
                              double* o, double* lse) {
  int n = tok_end > tok_begin ? tok_end - tok_begin : 0;
  exact_src S = {H, h, tok_begin, k_pool, v_pool, page_table};
  double qd[D_HEAD];
  int r = h * G + g;
  query_row(q, r, qd);
  attend_row(n, D_HEAD, qd, exact_key, exact_value, &S, 1.0 / sqrt((double)D_HEAD), o + (int64_t)r * D_HEAD,
             lse + r);
}

/* 8-bit-tier partial of query row g of KV head h [FMT, ATT] over pages
 * [page_begin, page_end): dequantise, then attend. */
static void partial_int8_row(int H, int G, int h, int g, const uint16_t* q, const uint8_t* rec_pool,
                             const int32_t* page_table8, int page_begin, int page_end, double* o, double* lse) {
  int np = page_end > page_begin ? page_end - page_begin : 0;
  int8_src S = {H, h, page_begin, rec_pool, page_table8};
  double qd[D_HEAD];
  int r = h * G + g;
  query_row(q, r, qd);
  attend_row(np * T_PAGE, D_HEAD, qd, int8_key, int8_value, &S, 1.0 / sqrt((double)D_HEAD),
             o + (int64_t)r * D_HEAD, lse + r);
}

/*
 * Integer query of one query row for one page [IQ]: q'_c = q_c * s_c in float32
 * (s in channel order), m = max_c |q'_c|; alpha = m / 127 and inv = 127 / m, each
 * one float32 division; qi_c = rint(q'_c * inv) (float32 product, half to even),
 * clamped to +-127.  m = 0 gives alpha = 0 and zero codes.  Returns alpha.
 */
float orc_query_codes(const uint16_t* q_row, const float* s, int8_t* qi) {
  float qp[D_HEAD];
  float m = 0.0f;
  for (int c = 0; c < D_HEAD; ++c) {
    qp[c] = bf16_float(q_row[c]) * s[c];
    float a = fabsf(qp[c]);
    if (a > m) m = a;
  }
  if (m == 0.0f) {
    for (int c = 0; c < D_HEAD; ++c) qi[c] = 0;
    return 0.0f;
  }
  const float inv = 127.0f / m;
  for (int c = 0; c < D_HEAD; ++c) {
    float y = rintf(qp[c] * inv);
    if (y > 127.0f) y = 127.0f;
    if (y < -127.0f) y = -127.0f;
    qi[c] = (int8_t)y;
  }
  return m / 127.0f;
}

/* 8-bit-tier partial of query row g with the integer query [IQ, FMT, ATT]: per
 * page the row's query is coded by orc_query_codes with the page's s_c, and
 *   score_t = scale * alpha * r_t * sum_c qi_c kc_tc   (the sum is exact);
 * values are dequantised (v = vc * u_c) and attended in double. */
static void partial_int8_iq_row(int H, int G, int h, int g, const uint16_t* q, const uint8_t* rec_pool,
                                const int32_t* page_table8, int page_begin, int page_end, double* o,
                                double* lse) {
  const int d = D_HEAD;
  const double scale = 1.0 / sqrt((double)d);
  int np = page_end > page_begin ? page_end - page_begin : 0;
  int n = np * T_PAGE;
  int8_src S = {H, h, page_begin, rec_pool, page_table8};
  double* sc = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
  const int r = h * G + g;
  for (int p = 0; p < np; ++p) {
    const uint8_t* rec = rec_pool + ((int64_t)page_table8[page_begin + p] * H + h) * REC_BYTES;
    const uint8_t* kc = rec + OFF_KC;
    float s[D_HEAD], rt[T_PAGE], s_stored[D_HEAD];
    memcpy(s_stored, rec + OFF_KS_CHAN, sizeof s_stored);
    for (int c = 0; c < D_HEAD; ++c) s[c] = s_stored[ks_pos(c)];
    memcpy(rt, rec + OFF_KS_TOK, sizeof rt);
    int8_t qi[D_HEAD];
    const float alpha = orc_query_codes(q + (int64_t)r * d, s, qi);
    for (int t = 0; t < T_PAGE; ++t) {
      int64_t dot = 0;
      for (int c = 0; c < d; ++c) dot += (int64_t)qi[c] * ((int)kc[kc_pos(t, c)] - 128);
      sc[p * T_PAGE + t] = scale * (double)alpha * (double)rt[t] * (double)dot;
    }
  }
  attend_scores(n, d, sc, int8_value, &S, o + (int64_t)r * d, lse + r);
  free(sc);
}

void orc_partial_exact(int H, int G, const uint16_t* q, const uint16_t* k_pool, const uint16_t* v_pool,
                       const int32_t* page_table, int tok_begin, int tok_end, double* o, double* lse) {
  for (int h = 0; h < H; ++h)
    for (int g = 0; g < G; ++g)
      partial_exact_row(H, G, h, g, q, k_pool, v_pool, page_table, tok_begin, tok_end, o, lse);
}

void orc_partial_int8(int H, int G, const uint16_t* q, const uint8_t* rec_pool, const int32_t* page_table8,
                      int page_begin, int page_end, double* o, double* lse) {
  for (int h = 0; h < H; ++h)
    for (int g = 0; g < G; ++g) partial_int8_row(H, G, h, g, q, rec_pool, page_table8, page_begin, page_end, o, lse);
}

void orc_partial_int8_iq(int H, int G, const uint16_t* q, const uint8_t* rec_pool, const int32_t* page_table8,
                         int page_begin, int page_end, double* o, double* lse) {
  for (int h = 0; h < H; ++h)
    for (int g = 0; g < G; ++g)
      partial_int8_iq_row(H, G, h, g, q, rec_pool, page_table8, page_begin, page_end, o, lse);
}

/*
 * Fold n_parts partials (o_i, lse_i) of `rows` rows [MERGE]:
 *   lse = ln sum_i exp(lse_i);  o = sum_i exp(lse_i - lse) o_i.
 * Partials with lse_i = -inf are skipped (their o_i is never read); if every
 * partial is empty the result is o = 0, lse = -inf.
 */
void orc_merge(int n_parts, int rows, int d, const double* o_parts, const double* lse_parts, double* o,
               double* lse) {
  for (int r = 0; r < rows; ++r) {
    double m = -INFINITY;
    for (int i = 0; i < n_parts; ++i) {
      double x = lse_parts[(int64_t)i * rows + r];
      if (x > m) m = x;
    }
    double* orow = o + (int64_t)r * d;
    for (int c = 0; c < d; ++c) orow[c] = 0.0;
    if (m == -INFINITY) {
      lse[r] = -INFINITY;
      continue;
    }
    double l = 0.0;
    for (int i = 0; i < n_parts; ++i) {
      double x = lse_parts[(int64_t)i * rows + r];
      if (x == -INFINITY) continue;
      l += exp(x - m);
    }
    double L = m + log(l);
    for (int i = 0; i < n_parts; ++i) {
      double x = lse_parts[(int64_t)i * rows + r];
      if (x == -INFINITY) continue;
      double w = exp(x - L);
      const double* oi = o_parts + ((int64_t)i * rows + r) * d;
      for (int c = 0; c < d; ++c) orow[c] += w * oi[c];
    }
    lse[r] = L;
  }
}

/* ====================================================== multi-request hybrid */

typedef struct {
  int B, H, G;
  const uint16_t *q, *k_pool, *v_pool;
  const uint8_t* rec_pool;
  const int32_t *page_table, *req_page_off, *n_exact_tokens;
  const int32_t *page_table8, *req_page_off8, *n_int8_pages;
  double *o, *lse;
  int int_query; /* 1: the 8-bit partials use the integer query [IQ] */
  int next;      /* next (request, head, query row) item, under the lock */
  pthread_mutex_t lock;
} hybrid_job;

/* Query row g of KV head h of request b: both tiers' partials of that row, folded
 * by orc_merge [TIERS, MERGE]. */
static void hybrid_item(hybrid_job* J, int item) {
  const int d = D_HEAD;
  const int G = J->G, rows = J->H * G;
  const int b = item / rows, h = (item % rows) / G, g = item % G;
  const int r = h * G + g;
  double* parts_o = (double*)malloc(sizeof(double) * 2 * (size_t)rows * d);
  double* parts_lse = (double*)malloc(sizeof(double) * 2 * (size_t)rows);
  const uint16_t* qb = J->q + (int64_t)b * rows * d;
  partial_exact_row(J->H, G, h, g, qb, J->k_pool, J->v_pool, J->page_table + J->req_page_off[b], 0,
                    J->n_exact_tokens[b], parts_o, parts_lse);
  (J->int_query ? partial_int8_iq_row : partial_int8_row)(J->H, G, h, g, qb, J->rec_pool,
                                                           J->page_table8 + J->req_page_off8[b], 0,
                                                           J->n_int8_pages[b], parts_o + (int64_t)rows * d,
                                                           parts_lse + rows);
  double po[2 * D_HEAD], pl[2];
  for (int i = 0; i < 2; ++i) {
    pl[i] = parts_lse[(int64_t)i * rows + r];
    memcpy(po + (int64_t)i * d, parts_o + ((int64_t)i * rows + r) * d, sizeof(double) * d);
  }
  orc_merge(2, 1, d, po, pl, J->o + ((int64_t)b * rows + r) * d, J->lse + (int64_t)b * rows + r);
  free(parts_o);
  free(parts_lse);
}

static void* hybrid_worker(void* arg) {
  hybrid_job* J = (hybrid_job*)arg;
  for (;;) {
    pthread_mutex_lock(&J->lock);
    int item = J->next++;
    pthread_mutex_unlock(&J->lock);
    if (item >= J->B * J->H * J->G) break;
    hybrid_item(J, item);
  }
  return 0;
}

/*
 * One hybrid decode step for B requests [TIERS]: per request and KV head, the
 * exact partial over the request's BF16 tokens [0, n_exact_tokens[b]) (CSR page
 * table page_table / req_page_off) and the 8-bit partial over its pages
 * [0, n_int8_pages[b]) (CSR page_table8 / req_page_off8), folded by orc_merge.
 * o is [B][H*G][256], lse is [B][H*G].  int_query = 1 takes the 8-bit partials
 * with the integer query.  Work is spread over n_threads threads by (request, KV
 * head, query row); the result does not depend on the thread count.
 */
void orc_hybrid_batched(int B, int H, int G, const uint16_t* q, const uint16_t* k_pool, const uint16_t* v_pool,
                        const uint8_t* rec_pool, const int32_t* page_table, const int32_t* req_page_off,
                        const int32_t* n_exact_tokens, const int32_t* page_table8, const int32_t* req_page_off8,
                        const int32_t* n_int8_pages, double* o, double* lse, int int_query, int n_threads) {
  hybrid_job J;
  J.B = B;
  J.H = H;
  J.G = G;
  J.q = q;
  J.k_pool = k_pool;
  J.v_pool = v_pool;
  J.rec_pool = rec_pool;
  J.page_table = page_table;
  J.req_page_off = req_page_off;
  J.n_exact_tokens = n_exact_tokens;
  J.page_table8 = page_table8;
  J.req_page_off8 = req_page_off8;
  J.n_int8_pages = n_int8_pages;
  J.o = o;
  J.lse = lse;
  J.int_query = int_query;
  J.next = 0;
  pthread_mutex_init(&J.lock, 0);
  if (n_threads < 1) n_threads = 1;
  if (n_threads > 256) n_threads = 256;
  pthread_t th[256];
  for (int i = 1; i < n_threads; ++i) pthread_create(&th[i], 0, hybrid_worker, &J);
  hybrid_worker(&J);
  for (int i = 1; i < n_threads; ++i) pthread_join(th[i], 0);
  pthread_mutex_destroy(&J.lock);
}
