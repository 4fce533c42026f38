// Page conversion: BF16 page-heads -> 8-bit records.
//
// "model quantization", section "An 8-bit page format shaped for its kernel":
// the key scale of a channel is the square root of its RMS over the page,
// normalised so the channel scales multiply to one and clamped to 2^+-14; a
// per-token-and-head factor covers the rest of the key's range; codes are
// symmetric in -127..127; values carry one scale per channel per page.
//
// One thread block converts one page-head (64 tokens x 256 channels of K and V):
//   1. the keys are bulk-copied into shared memory (the values, read twice, come
//      from global memory, so four blocks fit on an SM);
//   2. thread c owns channel c: u_c = max|v| / 127, and the key mean square with
//      compensated float32 additions of exact squares, as a rule in two chains of
//      32 (relative error below gamma_31^2 < 2^-38, or gamma_63^2 < 2^-36 for one
//      chain of 64: the bound of Ogita, Rump and Oishi's Sum2);
//   3. the geometric mean of the mean squares as a product of mantissas (float
//      pairs) and a sum of exponents, so the normalised fourth power x_c = ms_c / G
//      needs one multiplication; shat_c = x_c^(1/4); no double-precision arithmetic
//      anywhere (its rate on this GPU is a small fraction of FP32's);
//   4. the float32 neighbours of shat_c, found exactly (c^4 against x_c in
//      integer arithmetic); then warp 0 walks the channels (lane j holds 8
//      channels, the running log-error passes from lane to lane) choosing the
//      neighbour that keeps the running log-error of the product nearest zero,
//      while warps 1-7 write the value codes (channel-major, one 64-byte row per
//      channel), which need only u_c;
//   5. threads (token, quarter row) take y = k / s_c, the per-token absolute
//      maximum r_t = max|y| / 127 and the key codes, as rint of the correctly
//      rounded quotients (by reciprocal multiplication, with IEEE divisions
//      wherever that could differ).
// Fields are written at their swizzled positions (kc_byte, vc_byte, ks_index).
#include <cmath>

#include "common.cuh"

namespace tpk {

struct QSmem {
  alignas(128) uint16_t k[kPageTokens][kHeadDim];
  uint64_t bar;
  alignas(16) uint16_t vred[8][kHeadDim];  // per-warp maxima of |v| (bfloat16)
  float2 red_m[8];
  int red_e[8];
  float2 ig;  // 1 / G = (ig.x + ig.y) 2^ig_e
  int ig_e;
  alignas(16) float s[kHeadDim];
  alignas(16) float inv_s[kHeadDim];
  alignas(16) float u[kHeadDim];
  alignas(16) float slo[kHeadDim];
  alignas(16) float shi[kHeadDim];
  alignas(16) float dlo[kHeadDim];
  alignas(16) float dhi[kHeadDim];
  int bad;
};

// c^4 - x for a normal float c and x = mx 2^ex, mx an integer in (2^53.99, 2^55): the
// sign exactly, and the relative difference (c^4 - x) / x as a float estimate
// (rcp_xm: about 2^54 / mx).  With c = mc 2^ec (mc 24 bits), c^4 - x = 2^(4ec) (mc^4 -
// mx 2^s) for s = ex - 4ec; mc^4 < 2^96 is formed exactly in two 64-bit words, so the
// comparison is integer arithmetic only.  For c within a few ulp of x^(1/4), the
// only points evaluated, |c^4 - x| < 2^-19 x < 2^96 (bounds the magnitude's words).
struct Pow4Diff {
  int sign;
  float rel;
};
__device__ __forceinline__ Pow4Diff pow4_diff(float c, uint64_t mx, int ex, float rcp_xm) {
  const uint32_t cb = __float_as_uint(c);
  const uint64_t mc = (cb & 0x7fffffu) | 0x800000u;
  const int ec = (int)((cb >> 23) & 0xff) - 150;
  const int s = ex - 4 * ec;
  if (s <= 37) return {1, 1.f};    // mx 2^s < 2^92 <= mc^4
  if (s >= 43) return {-1, -1.f};  // mx 2^s > 2^96 > mc^4
  const uint64_t m2 = mc * mc;     // < 2^48
  const uint64_t p_lo = m2 * m2, p_hi = __umul64hi(m2, m2);
  const uint64_t q_lo = mx << s, q_hi = mx >> (64 - s);
  const uint64_t d_lo = p_lo - q_lo;
  const int64_t d_hi = (int64_t)(p_hi - q_hi - (p_lo < q_lo ? 1u : 0u));
  if (d_hi == 0 && d_lo == 0) return {0, 0.f};
  // |D| of D = d_hi 2^64 + d_lo (two's complement), then rel = D / (mx 2^s)
  uint64_t m_lo = d_lo, m_hi = (uint64_t)d_hi;
  if (d_hi < 0) {
    m_lo = ~d_lo + 1u;
    m_hi = ~(uint64_t)d_hi + (m_lo == 0 ? 1u : 0u);
  }
  const float mag = (float)(uint32_t)m_hi * 0x1p64f + (float)(uint32_t)(m_lo >> 32) * 0x1p32f + (float)(uint32_t)m_lo;
  const float rel = mag * rcp_xm * __int_as_float((127 - 54 - s) << 23);
  return {d_hi < 0 ? -1 : 1, d_hi < 0 ? -rel : rel};
}

// 2^k as a float, for -126 <= k <= 127
__device__ __forceinline__ float pow2f(int k) { return __uint_as_float((uint32_t)(k + 127) << 23); }
// the exponent of a positive normal float
__device__ __forceinline__ int expo(float x) { return (int)((__float_as_uint(x) >> 23) & 0xff) - 127; }

// The stored byte of a code: clamp(rint(q), -127, 127) + 128 (offset binary) for
// the quotient q = x / scale, correctly rounded.
__device__ __forceinline__ uint32_t quotient_byte(float q) {
  const float z = fminf(fmaxf(rintf(q), -127.f), 127.f);
  return (uint32_t)((int)z + 128);
}
__device__ __forceinline__ uint32_t code_byte(float x, float scale) {
  if (!(scale > 0.f)) return 128u;
  return quotient_byte(__fdiv_rn(x, scale));
}

// Codes by multiplication.  With inv = 1/scale correctly rounded, z = x * inv (a
// value) or x * inv_s * inv_r (a key) is within 6 * 2^-24 * |z| of the correctly
// rounded quotient (of the two correctly rounded divisions), i.e. within 2^-14.4
// for |z| <= 128, where all codes live.  rint(z) is then the code unless z lies
// within kCodeSlack (2^-12, a 4x margin) of a half-integer -- which happens
// often (an element equal to half its row's or channel's maximum gives exactly
// 63.5) -- so those bytes are rewritten from the divisions after the group is
// stored, as are all bytes of a scale outside [2^-100, 2^100].
constexpr float kCodeSlack = 0x1p-12f;
__device__ __forceinline__ bool near_half(float z) { return 0.5f - fabsf(z - rintf(z)) <= kCodeSlack; }

// ---- packed float pairs: one instruction does the FP32 work of two elements, which
// halves the issue slots of the arithmetic below (the kernel is bound by instruction
// issue).  b - a as fma(a, -1, b): the exact difference, rounded once, as a subtraction.
__device__ __forceinline__ float2 sub2(float2 b, float2 a) { return __ffma2_rn(a, make_float2(-1.f, -1.f), b); }
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// The magic number of the rounding below: for |z| <= 128, z + M lies in [2^23,
// 2^24), where float32 spacing is 1, so the sum rounds half to even exactly like
// rint (M is even), and the low byte of its encoding is (rint(z) + 128) mod 256,
// the stored byte.
constexpr float kRoundMagic = 12583040.f;  // 1.5 * 2^23 + 128
__device__ __forceinline__ bool fast_scale(float scale) { return scale >= 0x1p-100f && scale <= 0x1p100f; }

// Four codes of pages converted here (estimates within 127 (1 + 2^-20) in
// magnitude: the scales come from the maxima, so no clamp is needed) from an
// interval around each quotient estimate: the estimate x * w (w = 1/scale, or
// y * (1/r_t) for keys) lies within a relative 6 * 2^-24 of the correctly rounded
// quotient, so x * w widened by 2^-20 each way brackets it.  tA = x * w (1 + 2^-20)
// + M and tB = x * w (1 - 2^-20) + M, each one fused multiply-add rounded to an
// integer, agree iff rint is constant over the interval -- then it is the code;
// else (diff nonzero) the byte is redone by division.  The low byte of tA's
// encoding is the stored byte; four of them make one word.
constexpr float kIvHi = 1.f + 0x1p-20f, kIvLo = 1.f - 0x1p-20f;
__device__ __forceinline__ uint32_t code_word4_iv(float2 x01, float2 x23, float2 wa, float2 wb, uint32_t& diff,
                                                  float2 (&ta)[2], float2 (&tb)[2]) {
  const float2 m = make_float2(kRoundMagic, kRoundMagic);
  ta[0] = __ffma2_rn(x01, wa, m);
  ta[1] = __ffma2_rn(x23, wa, m);
  tb[0] = __ffma2_rn(x01, wb, m);
  tb[1] = __ffma2_rn(x23, wb, m);
  diff |= (__float_as_uint(ta[0].x) ^ __float_as_uint(tb[0].x));
  diff |= (__float_as_uint(ta[0].y) ^ __float_as_uint(tb[0].y));
  diff |= (__float_as_uint(ta[1].x) ^ __float_as_uint(tb[1].x));
  diff |= (__float_as_uint(ta[1].y) ^ __float_as_uint(tb[1].y));
  return __byte_perm(__byte_perm(__float_as_uint(ta[0].x), __float_as_uint(ta[0].y), 0x0040),
                     __byte_perm(__float_as_uint(ta[1].x), __float_as_uint(ta[1].y), 0x0040), 0x5410);
}
__device__ __forceinline__ uint32_t diff_bits4(const float2 (&ta)[2], const float2 (&tb)[2], int shift) {
  return ((uint32_t)(__float_as_uint(ta[0].x) != __float_as_uint(tb[0].x)) |
          ((uint32_t)(__float_as_uint(ta[0].y) != __float_as_uint(tb[0].y)) << 1) |
          ((uint32_t)(__float_as_uint(ta[1].x) != __float_as_uint(tb[1].x)) << 2) |
          ((uint32_t)(__float_as_uint(ta[1].y) != __float_as_uint(tb[1].y)) << 3)) << shift;
}

constexpr int kQuantThreads = 256;  // one thread per channel in the per-channel phases

// ---- float-float arithmetic on the FP32 pipe (GB300's FP64 rate is a small
// fraction of its FP32 rate): a value is hi + lo with |lo| about ulp(hi) / 2 or
// less.  Knuth's TwoSum and the FMA product error; the _rn intrinsics keep the
// compiler from contracting the error terms away.
struct DF {
  float hi, lo;
};
__device__ __forceinline__ DF df_fast_renorm(float s, float e) {  // |s| >= |e|
  const float h = __fadd_rn(s, e);
  return {h, __fsub_rn(e, __fsub_rn(h, s))};
}
__device__ __forceinline__ DF df_mul(DF a, DF b) {
  const float p = __fmul_rn(a.hi, b.hi);
  float e = fmaf(a.hi, b.hi, -p);
  e = __fadd_rn(e, __fadd_rn(__fmul_rn(a.hi, b.lo), __fmul_rn(a.lo, b.hi)));
  return df_fast_renorm(p, e);
}
__device__ __forceinline__ DF df_add(DF a, DF b) {
  const float s = __fadd_rn(a.hi, b.hi), bb = __fsub_rn(s, a.hi);
  const float e = __fadd_rn(__fadd_rn(__fsub_rn(a.hi, __fsub_rn(s, bb)), __fsub_rn(b.hi, bb)), __fadd_rn(a.lo, b.lo));
  const float h = __fadd_rn(s, e);  // s may be smaller than e after cancellation: full TwoSum
  const float hb = __fsub_rn(h, s);
  return {h, __fadd_rn(__fsub_rn(s, __fsub_rn(h, hb)), __fsub_rn(e, hb))};
}
// 2^(-i / 256), i = 0..255, as float pairs (filled from the host once per device)
__constant__ float2 c_pow2_neg[256];


__global__ void __launch_bounds__(kQuantThreads, 2) quantize_kernel(const __grid_constant__ QuantParams p) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  QSmem& S = *reinterpret_cast<QSmem*>(smem_raw);
  const int tid = threadIdx.x;
  const int i = blockIdx.x / p.H, h = blockIdx.x % p.H;
  const bool given = p.g_kchan != nullptr;

  if (tid == 0) {
    int64_t src = p.src[i], dst = p.dst[i];
    bool ok = src >= 0 && (p.kv_slots == 0 || src < p.kv_slots) && dst >= 0 && (p.rec_slots == 0 || dst < p.rec_slots);
    S.bad = ok ? 0 : 1;
    if (!ok) atomicOr(p.status, kStatusBadSlot);
    mbar_init(&S.bar, 1);
    fence_mbar_init();
    if (ok) {
      int64_t off = (src * p.H + h) * (int64_t)(kPageTokens * kHeadDim);
      mbar_arrive_expect_tx(&S.bar, kBf16PageHeadBytes);
      bulk_g2s(&S.k[0][0], p.k_pool + off, kBf16PageHeadBytes, &S.bar);
      // the values are read from global memory: start bringing them into L2 now
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p.v_pool + off), "r"(kBf16PageHeadBytes)
                   : "memory");
    }
  }
  __syncthreads();
  if (S.bad) return;
  const bool landed = mbar_wait(&S.bar, 0, p.status);
  if (__syncthreads_or(!landed)) return;

  uint8_t* rec = p.rec_pool + ((int64_t)p.dst[i] * p.H + h) * kRecordBytes;
  // values are read from global memory, twice (the maxima with 16-byte row loads,
  // then the codes, where a warp reads 32 neighbouring channels of one token and
  // hits L2), so only the keys occupy shared memory
  const uint16_t(*gv)[kHeadDim] = reinterpret_cast<const uint16_t(*)[kHeadDim]>(
      p.v_pool + ((int64_t)p.src[i] * p.H + h) * (int64_t)(kPageTokens * kHeadDim));
  const int64_t gidx = (int64_t)i * p.H + h;  // index into given-scale arrays
  const int c = tid;

  // value codes of channel ch, tokens t0 .. t0 + 15: 16 bytes of the channel's
  // 64-byte row (channel-major layout)
  // (t0 is a multiple of 16, so the 16 bytes are contiguous: vc_byte(ch, t0 + e) =
  // vc_byte(ch, t0) + e)
  auto value_codes = [&](int ch, int t0) {
    const float u = S.u[ch];
    const bool fast = fast_scale(u);
    const float inv = fast ? __frcp_rn(u) : 0.f;
    uint32_t redo = fast ? 0u : 0xffffu;
    uint32_t wv[4] = {0u, 0u, 0u, 0u};
    if (given) {  // scales from the caller: any magnitude, so clamp
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const float z = bf16_lo(__ldg(&gv[t0 + e][ch])) * inv;
        redo |= (uint32_t)near_half(z) << e;
        wv[e >> 2] |= quotient_byte(z) << (8 * (e & 3));
      }
    } else {
      const float2 wa = make_float2(inv * kIvHi, inv * kIvHi), wb = make_float2(inv * kIvLo, inv * kIvLo);
      float2 ta[4][2], tb[4][2];
      uint32_t diff = 0u;
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        const int t = t0 + 4 * g;
        const float2 x01 = make_float2(bf16_lo(__ldg(&gv[t][ch])), bf16_lo(__ldg(&gv[t + 1][ch])));
        const float2 x23 = make_float2(bf16_lo(__ldg(&gv[t + 2][ch])), bf16_lo(__ldg(&gv[t + 3][ch])));
        wv[g] = code_word4_iv(x01, x23, wa, wb, diff, ta[g], tb[g]);
      }
      if (diff) {  // rare: the interval holds a half-integer
#pragma unroll
        for (int g = 0; g < 4; ++g) redo |= diff_bits4(ta[g], tb[g], 4 * g);
      }
    }
    uint8_t* dst = rec + kOffVc + vc_byte(ch, t0);
    *reinterpret_cast<uint4*>(dst) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
    while (redo) {
      const int e = __ffs(redo) - 1;
      redo &= redo - 1;
      dst[e] = (uint8_t)code_byte(bf16_lo(__ldg(&gv[t0 + e][ch])), u);
    }
  };
  // (channel, 16-token quarter) items, channel fastest, so that a warp's lanes read
  // neighbouring channels of the same tokens
  constexpr int kValueItems = kHeadDim * kPageTokens / 16;

  if (given) {
    S.u[c] = p.g_vchan[gidx * kHeadDim + c];
    S.s[c] = p.g_kchan[gidx * kHeadDim + c];
    __syncthreads();
    for (int it = tid; it < kValueItems; it += kQuantThreads) value_codes(it & 255, (it >> 8) * 16);
  } else {
    // 2. thread c: u_c = max|v| / 127, and the key mean square: exact squares
    //    added with TwoSum into float pairs; the mean is kept as a normalised pair
    //    and an exponent (for step 4).
    //    A zero channel takes a = 2^-63, i.e. a mean square of 2^-252.
    {
      // value maxima: warp w reads rows w, w + 8, .., w + 56 with 16-byte loads (lane
      // l: channels 8l .. 8l + 7) and keeps the maxima of |v| as bfloat16 pairs (a
      // maximum is exact in any format; NaN is passed over, as by fmaxf); the
      // eight warps' maxima meet in shared memory after the next barrier
      const int l = tid & 31, w = tid >> 5;
      uint32_t m[4] = {0u, 0u, 0u, 0u};
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint4 x = __ldg(reinterpret_cast<const uint4*>(&gv[w + 8 * j][8 * l]));
        const uint32_t xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) asm("max.bf16x2 %0, %0, %1;" : "+r"(m[i]) : "r"(xs[i] & 0x7fff7fffu));
      }
      *reinterpret_cast<uint4*>(&S.vred[w][8 * l]) = make_uint4(m[0], m[1], m[2], m[3]);
    }
    // One pass over the key channel: max |k|, and the sum of squares in two TwoSum
    // chains (even and odd tokens) as packed pairs.  A square of a bfloat16 is exact
    // in float32 unless it underflows or overflows; for 2^-40 <= max|k| < 2^40 the sum
    // stays far below overflow and the underflowing squares (|k| < 2^-63) are below
    // 2^-60 of it, so the pair is used as is.  Outside that range the channel is
    // summed again scaled by 2^-e (e the exponent of max|k|), which makes every
    // square exact and below 1.
    float kmax = 0.f;
    float2 h2 = make_float2(0.f, 0.f), l2 = make_float2(0.f, 0.f);
#pragma unroll 8
    for (int t = 0; t < kPageTokens; t += 2) {
      const float2 kk = make_float2(bf16_lo(S.k[t][c]), bf16_lo(S.k[t + 1][c]));
      kmax = fmax3(kmax, fabsf(kk.x), fabsf(kk.y));
      const float2 sq = __fmul2_rn(kk, kk);
      const float2 sum = __fadd2_rn(h2, sq), bb = sub2(sum, h2);
      l2 = __fadd2_rn(l2, __fadd2_rn(sub2(h2, sub2(sum, bb)), sub2(sq, bb)));
      h2 = sum;
    }
    const bool kmax_pos = kmax > 0.f;
    float hsum = 0.f, lsum = 0.f;  // the sum of squares (scaled by 2^-2kexp), as a float pair
    int kexp = 0;
    if (kmax >= 0x1p-40f && kmax < 0x1p40f) {
      const DF sum = df_add(DF{h2.x, l2.x}, DF{h2.y, l2.y});
      hsum = sum.hi;
      lsum = sum.lo;
    } else if (kmax_pos) {
      frexpf(kmax, &kexp);
      const float sc = ldexpf(1.f, -kexp);  // kmax * sc in [0.5, 1) (2^-128 for the largest)
      for (int t = 0; t < kPageTokens; ++t) {
        const float y = bf16_lo(S.k[t][c]) * sc;
        const float sq = y * y;
        const float sum = hsum + sq, bb = sum - hsum;
        lsum += (hsum - (sum - bb)) + (sq - bb);
        hsum = sum;
      }
    }
    // 3. geometric mean G of ms over channels, as 1 / G: the product of the mean
    //    squares as a normalised float pair m (in [1, 2]) and an exponent sum E,
    //    multiplied in a shuffle tree; then 1 / G = (m 2^E)^(-1/256) = m^(-1/256)
    //    2^(-E/256), with m^(-1/256) by two Newton steps on z^256 m = 1 (seeded in
    //    float, each step squaring the error) and 2^(-E/256) = 2^-q 2^(-r/256), E =
    //    256 q + r, from a table.  Relative error about 2^-45, all on the FP32 pipe.
    //    ms_c = mc 2^Ec (mc a float pair in [1, 2)) is kept for step 4.
    DF mc;
    int Ec;
    if (kmax_pos) {
      mc = df_fast_renorm(hsum, lsum);
      const int k = expo(mc.hi);
      const float sc = pow2f(-k);
      mc = {mc.hi * sc, mc.lo * sc};
      Ec = 2 * kexp - 6 + k;  // the mean over 64 tokens: 2^-6
    } else {
      mc = {1.f, 0.f};  // 2^-252: a = 2^-63
      Ec = -252;
    }
    DF m = mc;
    int E = Ec;
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
      const DF mo = {__shfl_xor_sync(0xffffffffu, m.hi, off), __shfl_xor_sync(0xffffffffu, m.lo, off)};
      E += __shfl_xor_sync(0xffffffffu, E, off);
      m = df_mul(m, mo);
      if (m.hi >= 2.f) {
        m = {m.hi * 0.5f, m.lo * 0.5f};
        E += 1;
      }
    }
    if ((tid & 31) == 0) {
      S.red_m[tid >> 5] = make_float2(m.hi, m.lo);
      S.red_e[tid >> 5] = E;
    }
    __syncthreads();
    {
      float vmax = 0.f;
#pragma unroll
      for (int w = 0; w < 8; w += 2) vmax = fmax3(vmax, bf16_lo(S.vred[w][c]), bf16_lo(S.vred[w + 1][c]));
      S.u[c] = __fdiv_rn(vmax, 127.f);
    }
    if (tid == 0) {
      DF mm = {S.red_m[0].x, S.red_m[0].y};
      int ee = S.red_e[0];
      for (int w = 1; w < kQuantThreads / 32; ++w) {
        mm = df_mul(mm, DF{S.red_m[w].x, S.red_m[w].y});
        ee += S.red_e[w];
        if (mm.hi >= 2.f) {
          mm = {mm.hi * 0.5f, mm.lo * 0.5f};
          ee += 1;
        }
      }
      DF z = {exp2f(-log2f(mm.hi) * (1.f / kHeadDim)), 0.f};
      for (int it = 0; it < 2; ++it) {
        DF z256 = z;
#pragma unroll
        for (int sq = 0; sq < 8; ++sq) z256 = df_mul(z256, z256);
        const DF t = df_mul(z256, mm);                           // about 1
        DF d = df_add(DF{1.f, 0.f}, DF{-t.hi, -t.lo});           // 1 - m z^256
        d = {d.hi * (1.f / kHeadDim), d.lo * (1.f / kHeadDim)};  // (1 - m z^256) / 256
        z = df_add(z, df_mul(z, d));
      }
      const int q = (ee >= 0) ? ee / kHeadDim : -((-ee + kHeadDim - 1) / kHeadDim);
      const float2 w = c_pow2_neg[ee - kHeadDim * q];
      const DF inv = df_mul(z, DF{w.x, w.y});
      S.ig = make_float2(inv.hi, inv.lo);
      S.ig_e = -q;
    }
    __syncthreads();
    // 4. float32 neighbours of shat_c = (ms_c / G)^(1/4), clamped to 2^+-14.  A
    //    channel whose scale is fixed (clamped, or shat_c a float) gets lo = hi and
    //    zero log errors, so the walk keeps its running error unchanged there.
    {
      // x = ms_c / G = mc (1 / G) 2^(Ec + ig_e), as a float pair xm in [1, 2) and the
      // exponent X
      DF xm = df_mul(mc, DF{S.ig.x, S.ig.y});  // in (1/4, 2)
      int X = Ec + S.ig_e;
      {
        const int kx = expo(xm.hi);
        const float sc = pow2f(-kx);
        xm = {xm.hi * sc, xm.lo * sc};
        X += kx;
      }
      const bool at_pow2 = xm.hi == 1.f;  // x = 2^X (1 + xm.lo)
      float lo, hi, dl = 0.f, dh = 0.f;
      if (X > 56 || (X == 56 && !(at_pow2 && xm.lo < 0.f))) {  // x >= 2^56
        lo = hi = 0x1p14f;
      } else if (X < -56 || (X == -56 && at_pow2 && xm.lo <= 0.f)) {  // x <= 2^-56
        lo = hi = 0x1p-14f;
      } else {
        // x as an integer mantissa: mx = mh 2^31 + rint(xm.lo 2^54) with xm.hi = mh
        // 2^-23 (|xm.lo| <= 2^-24), x = mx 2^(X - 54) to within 2^-54 of x
        const uint32_t mh = (__float_as_uint(xm.hi) & 0x7fffffu) | 0x800000u;
        const uint64_t mx = (uint64_t)((int64_t)((uint64_t)mh << 31) + (int64_t)__float2int_rn(xm.lo * 0x1p54f));
        const int ex = X - 54;
        const float rcp_xm = __frcp_rn(xm.hi);
        // the square root of the square root of x rounded to float lies within 2 ulp
        // of shat: step from it, one neighbour at a time, to the bracket lo^4 <= x <
        // hi^4 (hi the successor of lo); two evaluations as a rule
        float cc = sqrtf(sqrtf(xm.hi * pow2f(X)));
        Pow4Diff dc = pow4_diff(cc, mx, ex, rcp_xm);
        float nb = cc;
        Pow4Diff dn = dc;
        if (dc.sign != 0) {
          const float dir = dc.sign > 0 ? 0.f : 0x1p127f;  // towards shat
          for (int it = 0; it < 4; ++it) {
            nb = nextafterf(cc, dir);
            dn = pow4_diff(nb, mx, ex, rcp_xm);
            if (dn.sign != dc.sign) break;  // shat lies between cc and nb (or at nb)
            cc = nb;
            dc = dn;
          }
        }
        if (dc.sign == 0 || dn.sign == 0) {
          lo = hi = dc.sign == 0 ? cc : nb;  // shat is a float
        } else {
          const bool up = dc.sign < 0;  // cc below shat, nb above
          lo = up ? cc : nb;
          hi = up ? nb : cc;
          // ln(c / shat) = ln(1 + a) / 4 for the relative error a of the fourth power
          const float a = up ? dc.rel : dn.rel, b = up ? dn.rel : dc.rel;
          dl = fmaf(-0.125f * a, a, 0.25f * a);
          dh = fmaf(-0.125f * b, b, 0.25f * b);
        }
      }
      S.slo[c] = lo;
      S.shi[c] = hi;
      S.dlo[c] = dl;
      S.dhi[c] = dh;
    }
    __syncthreads();
    if (tid < 32) {
      // 5. the compensated walk, sequential in the channels: lane j holds the
      //    candidates of channels 8j .. 8j + 7 in registers, and the running error
      //    E passes from lane to lane (every lane runs the same steps; lane j's
      //    result is kept)
      const int lane = tid;
      const float4 lo0 = *reinterpret_cast<const float4*>(&S.slo[8 * lane]);
      const float4 lo1 = *reinterpret_cast<const float4*>(&S.slo[8 * lane + 4]);
      const float4 hi0 = *reinterpret_cast<const float4*>(&S.shi[8 * lane]);
      const float4 hi1 = *reinterpret_cast<const float4*>(&S.shi[8 * lane + 4]);
      const float4 dl0 = *reinterpret_cast<const float4*>(&S.dlo[8 * lane]);
      const float4 dl1 = *reinterpret_cast<const float4*>(&S.dlo[8 * lane + 4]);
      const float4 dh0 = *reinterpret_cast<const float4*>(&S.dhi[8 * lane]);
      const float4 dh1 = *reinterpret_cast<const float4*>(&S.dhi[8 * lane + 4]);
      const float lo[8] = {lo0.x, lo0.y, lo0.z, lo0.w, lo1.x, lo1.y, lo1.z, lo1.w};
      const float hi[8] = {hi0.x, hi0.y, hi0.z, hi0.w, hi1.x, hi1.y, hi1.z, hi1.w};
      const float dl[8] = {dl0.x, dl0.y, dl0.z, dl0.w, dl1.x, dl1.y, dl1.z, dl1.w};
      const float dh[8] = {dh0.x, dh0.y, dh0.z, dh0.w, dh1.x, dh1.y, dh1.z, dh1.w};
      float sv[8];
      float E = 0.f;
      for (int j = 0; j < 32; ++j) {
        float Ej = E;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float a = Ej + dl[e], b = Ej + dh[e];
          const bool take_lo = fabsf(a) <= fabsf(b);
          if (lane == j) sv[e] = take_lo ? lo[e] : hi[e];
          Ej = take_lo ? a : b;
        }
        E = __shfl_sync(0xffffffffu, Ej, j);
      }
      *reinterpret_cast<float4*>(&S.s[8 * lane]) = make_float4(sv[0], sv[1], sv[2], sv[3]);
      *reinterpret_cast<float4*>(&S.s[8 * lane + 4]) = make_float4(sv[4], sv[5], sv[6], sv[7]);
    } else if (tid >= 32) {
      // meanwhile warps 1-7 write the value codes, which do not depend on s
      for (int it = tid - 32; it < kValueItems; it += kQuantThreads - 32) value_codes(it & 255, (it >> 8) * 16);
    }
  }
  __syncthreads();
  S.inv_s[c] = __frcp_rn(S.s[c]);
  // one flag for the block: every key channel scale is in the range where the
  // reciprocal estimates hold
  const bool s_fast = __syncthreads_and(fast_scale(S.s[c]));
  // ---- 5. codes: thread (token t, quarter q) handles 64 channels, chunks rotated
  //         by lane so that shared-memory reads do not conflict.  y_tc = k_tc / s_c
  //         is estimated as k * (1/s_c); the exact max |y| of the row comes from
  //         correctly rounded divisions of the elements whose estimate is within
  //         2^-20 of the estimated maximum (the argmax is among them).
  {
    const int t = tid >> 2, q = tid & 3, lane = tid & 31;
    // the estimates y = k * (1/s_c) of chunk k (8 channels, as 4 pairs); recomputed
    // in each pass, which costs less than holding 64 of them in registers
    auto estimates = [&](int k, float2(&y)[4]) {
      const int ch0 = q * 64 + ((k + lane) & 7) * 8;
      const uint4 w = *reinterpret_cast<const uint4*>(&S.k[t][ch0]);
      const float4 i0 = *reinterpret_cast<const float4*>(&S.inv_s[ch0]);
      const float4 i1 = *reinterpret_cast<const float4*>(&S.inv_s[ch0 + 4]);
      y[0] = __fmul2_rn(make_float2(bf16_lo(w.x), bf16_hi(w.x)), make_float2(i0.x, i0.y));
      y[1] = __fmul2_rn(make_float2(bf16_lo(w.y), bf16_hi(w.y)), make_float2(i0.z, i0.w));
      y[2] = __fmul2_rn(make_float2(bf16_lo(w.z), bf16_hi(w.z)), make_float2(i1.x, i1.y));
      y[3] = __fmul2_rn(make_float2(bf16_lo(w.w), bf16_hi(w.w)), make_float2(i1.z, i1.w));
    };
    // pass 1: the row maximum of the estimates, and a mask of the chunks whose
    // maximum lies within 2^-20 of the running maximum A when seen (all are dropped
    // when a chunk's maximum m has fl(m (1 - 2^-20)) > A).  Every chunk holding an
    // element >= thr = fl(amax (1 - 2^-20)) for the final row maximum amax is in
    // the mask: a chunk left out or dropped has its maximum below fl(a (1 - 2^-20))
    // for some running maximum a <= amax.  Only the marked chunks' elements are
    // then tested against thr and divided (the argmax is among them).
    float amax = 0.f;
    uint32_t chunks = 0u;
#pragma unroll 2
    for (int k = 0; k < 8; ++k) {
      float2 y[4];
      estimates(k, y);
      float cm = fmax3(fabsf(y[0].x), fabsf(y[0].y), fabsf(y[1].x));
      cm = fmax3(cm, fabsf(y[1].y), fabsf(y[2].x));
      cm = fmax3(cm, fabsf(y[2].y), fabsf(y[3].x));
      cm = fmaxf(cm, fabsf(y[3].y));
      if (cm * (1.f - 0x1p-20f) > amax) chunks = 0u;
      if (cm >= amax * (1.f - 0x1p-20f)) chunks |= 1u << k;
      amax = fmaxf(amax, cm);
    }
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    const float thr = amax * (1.f - 0x1p-20f);
    if (!s_fast) chunks = 0xffu;
    float ymax = 0.f;
    while (chunks) {
      const int k = __ffs(chunks) - 1;
      chunks &= chunks - 1;
      const int ch0 = q * 64 + ((k + lane) & 7) * 8;
      for (int e = 0; e < 8; ++e) {
        const float kv = bf16_lo(S.k[t][ch0 + e]);
        if (!s_fast || fabsf(kv * S.inv_s[ch0 + e]) >= thr)
          ymax = fmaxf(ymax, fabsf(__fdiv_rn(kv, S.s[ch0 + e])));
      }
    }
    ymax = fmaxf(ymax, __shfl_xor_sync(0xffffffffu, ymax, 1));
    ymax = fmaxf(ymax, __shfl_xor_sync(0xffffffffu, ymax, 2));
    const float r = given ? p.g_ktok[gidx * kPageTokens + t] : __fdiv_rn(ymax, 127.f);
    const bool fast = s_fast && fast_scale(r);
    const float inv_r = fast ? __frcp_rn(r) : 0.f;
    const float2 ra = make_float2(inv_r * kIvHi, inv_r * kIvHi), rb = make_float2(inv_r * kIvLo, inv_r * kIvLo);
    uint8_t* kc = rec + kOffKc;
#pragma unroll 2
    for (int k = 0; k < 8; ++k) {
      float2 y[4];
      estimates(k, y);
      const int ch0 = q * 64 + ((k + lane) & 7) * 8;
      uint32_t wk[2] = {0u, 0u};
      uint32_t redo = fast ? 0u : 0xffu;
      if (given) {  // r from the caller: any magnitude, so clamp
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float z = ((e & 1) ? y[e >> 1].y : y[e >> 1].x) * inv_r;
          redo |= (uint32_t)near_half(z) << e;
          wk[e >> 2] |= quotient_byte(z) << (8 * (e & 3));
        }
      } else {
        float2 ta[2][2], tb[2][2];
        uint32_t diff = 0u;
        wk[0] = code_word4_iv(y[0], y[1], ra, rb, diff, ta[0], tb[0]);
        wk[1] = code_word4_iv(y[2], y[3], ra, rb, diff, ta[1], tb[1]);
        if (diff) {  // rare
          redo |= diff_bits4(ta[0], tb[0], 0) | diff_bits4(ta[1], tb[1], 4);
        }
      }
      // (ch0 is a multiple of 8: kc_byte(t, ch0 + e) = kc_byte(t, ch0) + e)
      uint8_t* dst = kc + kc_byte(t, ch0);
      *reinterpret_cast<uint2*>(dst) = make_uint2(wk[0], wk[1]);
      while (redo) {
        const int e = __ffs(redo) - 1;
        redo &= redo - 1;
        dst[e] = (uint8_t)code_byte(__fdiv_rn(bf16_lo(S.k[t][ch0 + e]), S.s[ch0 + e]), r);
      }
    }
    if (q == 0) reinterpret_cast<float*>(rec + kOffKsTok)[t] = r;
  }
  reinterpret_cast<float*>(rec + kOffKsChan)[ks_index(c)] = S.s[c];
  reinterpret_cast<float*>(rec + kOffVsChan)[c] = S.u[c];
}

cudaError_t launch_quantize(const QuantParams& p, int n_pages, cudaStream_t stream) {
  static DeviceOnce once;
  const int smem = (int)sizeof(QSmem);
  const cudaError_t e = once.run([&] {
    cudaError_t r = cudaFuncSetAttribute(quantize_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (r != cudaSuccess) return r;
    float2 t[256];  // 2^(-i/256) split into float pairs
    for (int i = 0; i < 256; ++i) {
      const double v = std::exp2(-i / 256.0);
      const float hi = (float)v;
      t[i] = make_float2(hi, (float)(v - (double)hi));
    }
    return cudaMemcpyToSymbol(c_pow2_neg, t, sizeof t);
  });
  if (e != cudaSuccess) return e;
  if (n_pages == 0) return cudaSuccess;
  quantize_kernel<<<n_pages * p.H, kQuantThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace tpk
