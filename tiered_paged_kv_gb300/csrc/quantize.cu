// Page conversion: BF16 page-heads -> 8-bit records.
//
// "model quantization", section "An 8-bit page format shaped for its kernel":
// the key scale of a channel is the square root of its RMS over the page,
// normalised so the channel scales multiply to one and clamped to 2^+-14; a
// per-token-and-head factor covers the rest of the key's range; codes are
// symmetric in -127..127; values carry one scale per channel per page.
//
// One thread block converts one page-head (64 tokens x 256 channels of K and V):
//   1. the page-head is bulk-copied into shared memory;
//   2. thread c owns channel c: the key channel's mean square is accumulated
//      exactly (bfloat16 squares summed as 64-bit fixed point), the value
//      channel's absolute maximum gives u_c = max|v| / 127;
//   3. the geometric mean of the mean squares is formed as a product of
//      mantissas (double) and a sum of exponents, so the normalised fourth power
//      x_c = ms_c / G needs one multiplication; shat_c = x_c^(1/4);
//   4. the float32 neighbours of shat_c are found exactly (c^4 against x_c with
//      an FMA-exact product), and one thread walks the channels choosing the
//      neighbour that keeps the running log-error of the product nearest zero,
//      while the other seven warps write the value codes (they need only u_c);
//   5. threads (token, quarter row) divide keys by s_c, take the per-token
//      absolute maximum r_t = max|y| / 127 and form the codes with IEEE float32
//      divisions and half-to-even rint.  Value codes are stored channel-major
//      (one 64-byte row per channel).  Fields are written at their swizzled
//      positions (kc_byte, vc_byte, ks_index).
#include "common.cuh"

namespace tpk {

struct QSmem {
  alignas(128) uint16_t k[kPageTokens][kHeadDim];
  alignas(128) uint16_t v[kPageTokens][kHeadDim];
  uint64_t bar;
  double red_m[8];
  int red_e[8];
  double invG;
  alignas(16) float s[kHeadDim];
  alignas(16) float u[kHeadDim];
  alignas(16) float slo[kHeadDim];
  alignas(16) float shi[kHeadDim];
  alignas(16) float dlo[kHeadDim];
  alignas(16) float dhi[kHeadDim];
  alignas(16) int exact[kHeadDim];
  int bad;
};

// c^4 - x, with c^2 exact in double and c^4 = hi + lo exact by FMA.
__device__ __forceinline__ double pow4_minus(float c, double x) {
  double c2 = (double)c * (double)c;
  double hi = c2 * c2;
  double lo = fma(c2, c2, -hi);
  return (hi - x) + lo;
}

// The stored byte of a code: clamp(rint(x / scale), -127, 127) + 128 (offset binary).
__device__ __forceinline__ uint32_t code_byte(float x, float scale) {
  if (!(scale > 0.f)) return 128u;
  float z = rintf(__fdiv_rn(x, scale));
  z = fminf(fmaxf(z, -127.f), 127.f);
  return (uint32_t)((int)z + 128);
}

constexpr int kQuantThreads = 256;  // one thread per channel in the per-channel phases

__global__ void __launch_bounds__(kQuantThreads) quantize_kernel(const __grid_constant__ QuantParams p) {
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
      mbar_arrive_expect_tx(&S.bar, 2 * kBf16PageHeadBytes);
      bulk_g2s(&S.k[0][0], p.k_pool + off, kBf16PageHeadBytes, &S.bar);
      bulk_g2s(&S.v[0][0], p.v_pool + off, kBf16PageHeadBytes, &S.bar);
    }
  }
  __syncthreads();
  if (S.bad) return;
  const bool landed = mbar_wait(&S.bar, 0, p.status);
  if (__syncthreads_or(!landed)) return;

  uint8_t* rec = p.rec_pool + ((int64_t)p.dst[i] * p.H + h) * kRecordBytes;
  const int64_t gidx = (int64_t)i * p.H + h;  // index into given-scale arrays
  const int c = tid;

  // ---- 2. per-channel statistics
  {
    float vmax = 0.f;
    for (int t = 0; t < kPageTokens; ++t) vmax = fmaxf(vmax, fabsf(bf16_lo(S.v[t][c])));
    S.u[c] = given ? p.g_vchan[gidx * kHeadDim + c] : __fdiv_rn(vmax, 127.f);
  }
  // value codes of channel ch, tokens t0 .. t0 + 15: 16 bytes of the channel's
  // 64-byte row (channel-major layout)
  auto value_codes = [&](int ch, int t0) {
    const float u = S.u[ch];
    uint32_t wv[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int e = 0; e < 16; ++e) wv[e >> 2] |= code_byte(bf16_lo(S.v[t0 + e][ch]), u) << (8 * (e & 3));
    *reinterpret_cast<uint4*>(rec + kOffVc + vc_byte(ch, t0)) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
  };
  double mant = 1.0;
  int expo = 0;
  double ms = 0.0;
  if (!given) {
    int emax = 1;
    for (int t = 0; t < kPageTokens; ++t) {
      int e = (S.k[t][c] >> 7) & 0xff;
      emax = max(emax, e);
    }
    // element = m * 2^(e - 134) (m with the hidden bit; subnormals use e = 1);
    // square = m^2 * 2^(2e - 268); fixed point unit 2^(2 emax - 308)
    unsigned long long acc = 0;
    for (int t = 0; t < kPageTokens; ++t) {
      uint32_t bits = S.k[t][c] & 0x7fffu;
      int e = bits >> 7;
      uint32_t m = bits & 0x7fu;
      if (e) m |= 0x80u; else e = 1;
      unsigned long long m2 = (unsigned long long)(m * m);
      int sh = 2 * (emax - e);
      if (sh <= 40) acc += m2 << (40 - sh);
      else if (sh < 56) acc += m2 >> (sh - 40);
    }
    ms = acc ? ldexp((double)acc, 2 * emax - 308 - 6) : 0x1p-252;  // mean over 64 tokens
    mant = frexp(ms, &expo);
  }
  // ---- 3. geometric mean of ms over channels: product of mantissas, sum of exponents
  if (!given) {
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
      double mo = __shfl_xor_sync(0xffffffffu, mant, off);
      int eo = __shfl_xor_sync(0xffffffffu, expo, off);
      int t;
      mant = frexp(mant * mo, &t);
      expo += eo + t;
    }
    if ((tid & 31) == 0) {
      S.red_m[tid >> 5] = mant;
      S.red_e[tid >> 5] = expo;
    }
  }
  __syncthreads();
  if (!given && tid == 0) {
    double m = S.red_m[0];
    int e = S.red_e[0];
    for (int w = 1; w < 8; ++w) {
      int t;
      m = frexp(m * S.red_m[w], &t);
      e += S.red_e[w] + t;
    }
    double lnG = (log(m) + (double)e * 0.69314718055994530942) / kHeadDim;
    S.invG = exp(-lnG);
  }
  __syncthreads();
  // ---- 4. float32 neighbours of shat_c = (ms_c / G)^(1/4), clamped to 2^+-14
  if (!given) {
    double x = ms * S.invG;
    float lo, hi, dl = 0.f, dh = 0.f;
    int ex = 0;
    if (x >= 0x1p56) {
      lo = hi = 0x1p14f;
      ex = 1;
    } else if (x <= 0x1p-56) {
      lo = hi = 0x1p-14f;
      ex = 1;
    } else {
      float cc = sqrtf(sqrtf((float)x));
      for (int it = 0; it < 4; ++it) {
        if (pow4_minus(cc, x) > 0.0) cc = nextafterf(cc, 0.f);
        else if (pow4_minus(nextafterf(cc, 0x1p127f), x) <= 0.0) cc = nextafterf(cc, 0x1p127f);
        else break;
      }
      double df = pow4_minus(cc, x);
      if (df == 0.0) {
        lo = hi = cc;
        ex = 1;
      } else {
        lo = cc;
        hi = nextafterf(cc, 0x1p127f);
        double rx = 1.0 / x;
        double a = df * rx, b = pow4_minus(hi, x) * rx;  // relative error of the fourth power
        dl = (float)(0.25 * a - 0.125 * a * a);           // ln(lo / shat)
        dh = (float)(0.25 * b - 0.125 * b * b);           // ln(hi / shat)
      }
    }
    S.slo[c] = lo;
    S.shi[c] = hi;
    S.dlo[c] = dl;
    S.dhi[c] = dh;
    S.exact[c] = ex;
  }
  __syncthreads();
  if (given) {
    S.s[c] = p.g_kchan[gidx * kHeadDim + c];
    for (int t0 = 0; t0 < kPageTokens; t0 += 16) value_codes(c, t0);
  } else if (tid < 32) {
    // The compensated walk is sequential in the channels; one lane runs it with
    // each group of 8 channels' candidates loaded into registers first, while the
    // other seven warps write the value codes, which do not depend on s.
    if (tid == 0) {
      float E = 0.f;
      for (int ch0 = 0; ch0 < kHeadDim; ch0 += 8) {
        float lo[8], hi[8], dl[8], dh[8], sv[8];
        int ex[8];
        *reinterpret_cast<float4*>(lo) = *reinterpret_cast<const float4*>(&S.slo[ch0]);
        *reinterpret_cast<float4*>(lo + 4) = *reinterpret_cast<const float4*>(&S.slo[ch0 + 4]);
        *reinterpret_cast<float4*>(hi) = *reinterpret_cast<const float4*>(&S.shi[ch0]);
        *reinterpret_cast<float4*>(hi + 4) = *reinterpret_cast<const float4*>(&S.shi[ch0 + 4]);
        *reinterpret_cast<float4*>(dl) = *reinterpret_cast<const float4*>(&S.dlo[ch0]);
        *reinterpret_cast<float4*>(dl + 4) = *reinterpret_cast<const float4*>(&S.dlo[ch0 + 4]);
        *reinterpret_cast<float4*>(dh) = *reinterpret_cast<const float4*>(&S.dhi[ch0]);
        *reinterpret_cast<float4*>(dh + 4) = *reinterpret_cast<const float4*>(&S.dhi[ch0 + 4]);
        *reinterpret_cast<int4*>(ex) = *reinterpret_cast<const int4*>(&S.exact[ch0]);
        *reinterpret_cast<int4*>(ex + 4) = *reinterpret_cast<const int4*>(&S.exact[ch0 + 4]);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float a = E + dl[e], b = E + dh[e];
          const bool take_lo = ex[e] || fabsf(a) <= fabsf(b);
          sv[e] = take_lo ? lo[e] : hi[e];
          E = ex[e] ? E : (take_lo ? a : b);
        }
        *reinterpret_cast<float4*>(&S.s[ch0]) = *reinterpret_cast<const float4*>(sv);
        *reinterpret_cast<float4*>(&S.s[ch0 + 4]) = *reinterpret_cast<const float4*>(sv + 4);
      }
    }
  } else {
    // (channel, 16-token quarter) items spread evenly over the seven warps
    for (int it = tid - 32; it < kHeadDim * 4; it += kQuantThreads - 32) value_codes(it >> 2, (it & 3) * 16);
  }
  __syncthreads();
  // ---- 5. codes: thread (token t, quarter q) handles 64 channels, chunks rotated
  //         by lane so that shared-memory reads do not conflict
  {
    const int t = tid >> 2, q = tid & 3, lane = tid & 31;
    float y[8][8];
    float ymax = 0.f;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int ch0 = q * 64 + ((k + lane) & 7) * 8;
      uint4 w = *reinterpret_cast<const uint4*>(&S.k[t][ch0]);
      float f[8] = {bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y),
                    bf16_lo(w.z), bf16_hi(w.z), bf16_lo(w.w), bf16_hi(w.w)};
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        y[k][e] = __fdiv_rn(f[e], S.s[ch0 + e]);
        ymax = fmaxf(ymax, fabsf(y[k][e]));
      }
    }
    ymax = fmaxf(ymax, __shfl_xor_sync(0xffffffffu, ymax, 1));
    ymax = fmaxf(ymax, __shfl_xor_sync(0xffffffffu, ymax, 2));
    const float r = given ? p.g_ktok[gidx * kPageTokens + t] : __fdiv_rn(ymax, 127.f);
    uint8_t* kc = rec + kOffKc;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int ch0 = q * 64 + ((k + lane) & 7) * 8;
      uint32_t wk[2] = {0u, 0u};
#pragma unroll
      for (int e = 0; e < 8; ++e) wk[e >> 2] |= code_byte(y[k][e], r) << (8 * (e & 3));
      *reinterpret_cast<uint2*>(kc + kc_byte(t, ch0)) = make_uint2(wk[0], wk[1]);
    }
    if (q == 0) reinterpret_cast<float*>(rec + kOffKsTok)[t] = r;
  }
  reinterpret_cast<float*>(rec + kOffKsChan)[ks_index(c)] = S.s[c];
  reinterpret_cast<float*>(rec + kOffVsChan)[c] = S.u[c];
}

cudaError_t launch_quantize(const QuantParams& p, int n_pages, cudaStream_t stream) {
  static bool configured = false;
  const int smem = (int)sizeof(QSmem);
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(quantize_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  if (n_pages == 0) return cudaSuccess;
  quantize_kernel<<<n_pages * p.H, kQuantThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace tpk
