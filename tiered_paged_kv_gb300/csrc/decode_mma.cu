// Split-tier paged decode attention on the tensor cores (mma.sync).
//
// One thread block = one unit (a range of pages of one tier for one (request,
// KV head)).  A producer warp streams the unit's items into a ring of 6
// shared-memory slots; 4 consumer warps each take whole items (item j goes to
// warp j % 4) and keep their own online-softmax state and FP32 output for the 8
// query rows of the GQA group.  Thread (g, t) = (lane / 4, lane % 4) of a
// consumer warp owns query row g and output channels 8n + 2t + {0, 1}.
//
// 8-bit tier ("SYCL", "Attention that reads 8-bit history"): both products run on
// the integer tensor path (mma m16n8k32 s8 x s8 -> s32), reading the page's codes
// straight from shared memory:
//   QK  A = the folded query q'_c = q_c s_c (per page) quantised per row to a
//         high and a low int8 plane (rows 0-7 and 8-15 of the 16-row tile:
//         q' ~ sigma (hi + lo / 254)), B = the key codes; the per-token factor
//         r_t is applied after the dot product;
//   PV  A = the probabilities as int8 high/low planes (p ~ (hi + lo / 254) / 127),
//         B = the value codes (channel-major, four consecutive tokens per word);
//         the page's integer result is rescaled by the value scale u_c and added
//         to the FP32 accumulator once per page.
// Exact tier: BF16 half-pages (32 tokens) staged with a padded row pitch so
// ldmatrix reads are conflict-free; QK on bf16 mma with q exact; P enters PV as
// bf16 high/low planes (rows 0-7 / 8-15), giving about 16 bits of P.
//
// Online softmax ("SYCL", "Exact tricks and a two-owner decoder"): the running
// maximum is an integer in base 2, every rescale is a power of two built by
// exponent arithmetic, and the rescale is skipped when all eight rows' factors
// are 1 (a warp vote).
#include "decode_common.cuh"

namespace tpk {

constexpr int kMmaCons = kDecWarps;              // consumer warps
constexpr int kMmaThreads = (kMmaCons + 1) * 32;  // + one producer warp
constexpr int kMmaSlots = 6;
constexpr int kPad = 528;  // BF16 row pitch in shared memory (512 B + 16 B)
constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23: float + kMagic rounds to an integer in the low bits
constexpr unsigned kAll = 0xffffffffu;

struct MmaSmem {
  alignas(128) uint8_t slot[kMmaSlots][kSlotBytes];
  uint64_t full[kMmaSlots];
  uint64_t empty[kMmaSlots];
  int valid[kMmaSlots];
  int pt[kPtCache];
  alignas(16) uint32_t q[kGroup][kHeadDim / 2];  // the unit's query rows (bf16 pairs)
  float ep_m[kDecWarps][kGroup];
  float ep_l[kDecWarps][kGroup];
  int is_last;
  int abort;
};

// ----------------------------------------------------------------- PTX
__device__ __forceinline__ void mma_s8(int (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+r"(d[0]), "+r"(d[1]), "+r"(d[2]), "+r"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p))
               : "memory");
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p))
               : "memory");
}

// low bytes of four words -> one word
__device__ __forceinline__ uint32_t pack4(uint32_t b0, uint32_t b1, uint32_t b2, uint32_t b3) {
  return __byte_perm(__byte_perm(b0, b1, 0x0040), __byte_perm(b2, b3, 0x0040), 0x5410);
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// ----------------------------------------------------------------- producer
__device__ __forceinline__ void mma_issue(const DecodeParams& p, const UnitInfo& ui, const Items& it, MmaSmem& S,
                                          int j, int s) {
  int page = item_page(ui, it, j);
  int idx = page - it.pg_first;
  int64_t slot = idx < kPtCache ? S.pt[idx]
                                : __ldg((ui.tier == 0 ? p.page_table : p.page_table8) + ui.pt_off + page);
  int64_t lim = ui.tier == 0 ? p.kv_slots : p.rec_slots;
  bool ok = slot >= 0 && (lim == 0 || slot < lim);
  S.valid[s] = ok ? 1 : 0;
  if (!ok) {
    atomicOr(p.status, kStatusBadSlot);
    mbar_arrive(&S.full[s]);
    return;
  }
  if (ui.tier == 0) {
    const int half = (it.first + j) & 1;
    const int64_t off = ((slot * p.H + ui.h) * kPageTokens + half * 32) * (int64_t)kHeadDim;
    mbar_arrive_expect_tx(&S.full[s], 32768);
    for (int r = 0; r < 32; ++r) {
      bulk_g2s(S.slot[s] + r * kPad, p.k_pool + off + r * kHeadDim, 512, &S.full[s]);
      bulk_g2s(S.slot[s] + (32 + r) * kPad, p.v_pool + off + r * kHeadDim, 512, &S.full[s]);
    }
  } else {
    const uint8_t* src = p.rec_pool + (slot * p.H + ui.h) * (int64_t)kRecordBytes;
    mbar_arrive_expect_tx(&S.full[s], kRecordBytes);
    bulk_g2s(S.slot[s], src, kRecordBytes, &S.full[s]);
  }
}

// Online-softmax update for one item: x[] are this thread's base-2 scores (row
// g), -inf where masked.  Rescales O when the row maximum moved (skipped when
// all rows keep their maximum) and turns x[] into weights.
template <int N>
__device__ __forceinline__ void softmax_update(float (&x)[N], float& m_run, float& l_run, float (&O)[32][2]) {
  float mx = kNegInf;
#pragma unroll
  for (int i = 0; i < N; ++i) mx = fmaxf(mx, x[i]);
  mx = fmaxf(mx, __shfl_xor_sync(kAll, mx, 1));
  mx = fmaxf(mx, __shfl_xor_sync(kAll, mx, 2));
  const float m_new = (mx == kNegInf) ? m_run : fmaxf(m_run, ceilf(mx));
  const float alpha = (m_new == m_run) ? 1.f : (m_run == kNegInf ? 0.f : ldexpf(1.f, (int)(m_run - m_new)));
  if (!__all_sync(kAll, alpha == 1.f)) {
#pragma unroll
    for (int n = 0; n < 32; ++n) {
      O[n][0] *= alpha;
      O[n][1] *= alpha;
    }
  }
  float l = l_run * alpha;
#pragma unroll
  for (int i = 0; i < N; ++i) {
    x[i] = (x[i] == kNegInf) ? 0.f : exp2f(x[i] - m_new);
    l += x[i];
  }
  l_run = l;
  m_run = m_new;
}

// ---------------------------------------------------------------- 8-bit page
__device__ __forceinline__ void process_int8_page(const uint8_t* rec, const uint32_t* qrow, float qscale,
                                                  float& m_run, float& l_run, float (&O)[32][2]) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const float* ks = reinterpret_cast<const float*>(rec + kOffKsChan);
  const float* kr = reinterpret_cast<const float*>(rec + kOffKsTok);
  const float* vs = reinterpret_cast<const float*>(rec + kOffVsChan);

  // q'_c = q_c s_c for this thread's 64 channels 64J + 16t + i of row g
  float amax = 0.f;
#pragma unroll
  for (int J = 0; J < 4; ++J) {
    uint32_t qb[8];
    {
      uint4 a = *reinterpret_cast<const uint4*>(qrow + 32 * J + 8 * t);
      uint4 b = *reinterpret_cast<const uint4*>(qrow + 32 * J + 8 * t + 4);
      qb[0] = a.x; qb[1] = a.y; qb[2] = a.z; qb[3] = a.w; qb[4] = b.x; qb[5] = b.y; qb[6] = b.z; qb[7] = b.w;
    }
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      float4 s4 = *reinterpret_cast<const float4*>(ks + 64 * J + 16 * t + 4 * v);
      uint32_t w0 = qb[2 * v], w1 = qb[2 * v + 1];
      amax = fmaxf(amax, fabsf(bf16_lo(w0) * s4.x));
      amax = fmaxf(amax, fabsf(bf16_hi(w0) * s4.y));
      amax = fmaxf(amax, fabsf(bf16_lo(w1) * s4.z));
      amax = fmaxf(amax, fabsf(bf16_hi(w1) * s4.w));
    }
  }
  amax = fmaxf(amax, __shfl_xor_sync(kAll, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(kAll, amax, 2));
  const float inv = amax > 0.f ? 127.f / amax : 0.f;
  const float arow = amax > 0.f ? qscale * (amax * (1.f / 127.f)) * (1.f / 254.f) : 0.f;

  // int8 planes of q': A fragments for the 8 k-steps of 32 channels
  uint32_t qa[8][4];
#pragma unroll
  for (int J = 0; J < 4; ++J) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint32_t hi[8], lo[8];
      const uint4 qv = *reinterpret_cast<const uint4*>(qrow + 32 * J + 8 * t + 4 * h);
      const uint32_t qh[4] = {qv.x, qv.y, qv.z, qv.w};
#pragma unroll
      for (int v = 0; v < 2; ++v) {
        float4 s4 = *reinterpret_cast<const float4*>(ks + 64 * J + 16 * t + 8 * h + 4 * v);
        uint32_t w0 = qh[2 * v], w1 = qh[2 * v + 1];
        float x[4] = {bf16_lo(w0) * s4.x, bf16_hi(w0) * s4.y, bf16_lo(w1) * s4.z, bf16_hi(w1) * s4.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float t1 = fmaf(x[e], inv, kMagic);
          float hf = t1 - kMagic;
          float res = fmaf(x[e], inv, -hf);
          float t2 = fmaf(res, 254.f, kMagic);
          hi[4 * v + e] = __float_as_uint(t1);
          lo[4 * v + e] = __float_as_uint(t2);
        }
      }
      qa[2 * J + h][0] = pack4(hi[0], hi[1], hi[2], hi[3]);
      qa[2 * J + h][1] = pack4(lo[0], lo[1], lo[2], lo[3]);
      qa[2 * J + h][2] = pack4(hi[4], hi[5], hi[6], hi[7]);
      qa[2 * J + h][3] = pack4(lo[4], lo[5], lo[6], lo[7]);
    }
  }

  // QK: n-tile j holds keys 16 (n / 2) + 2 j + (n & 1) in column n, so thread t
  // receives the scores of keys 16 t + 2 j + {0, 1}.
  float x[16];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint8_t* krow = rec + kOffKc + (16 * (g >> 1) + 2 * j + (g & 1)) * kHeadDim + 16 * t;
    int c[4] = {0, 0, 0, 0};
#pragma unroll
    for (int J = 0; J < 4; ++J) {
      uint4 w = *reinterpret_cast<const uint4*>(krow + 64 * J);
      mma_s8(c, qa[2 * J], w.x, w.y);
      mma_s8(c, qa[2 * J + 1], w.z, w.w);
    }
    x[2 * j] = (float)(c[0] * 254 + c[2]);
    x[2 * j + 1] = (float)(c[1] * 254 + c[3]);
  }
  // per-token factor r_t after the dot product (keys 16t .. 16t+15 of this thread)
#pragma unroll
  for (int v = 0; v < 4; ++v) {
    float4 r4 = *reinterpret_cast<const float4*>(kr + 16 * t + 4 * v);
    x[4 * v] *= arow * r4.x;
    x[4 * v + 1] *= arow * r4.y;
    x[4 * v + 2] *= arow * r4.z;
    x[4 * v + 3] *= arow * r4.w;
  }
  softmax_update<16>(x, m_run, l_run, O);

  // P as int8 planes: k-step s covers keys 16 t + 8 s + (0..7) of thread t
  uint32_t pa[2][4];
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    uint32_t hi[8], lo[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      float v = 127.f * x[8 * s + e];
      float t1 = v + kMagic;
      float hf = t1 - kMagic;
      float t2 = fmaf(v - hf, 254.f, kMagic);
      hi[e] = __float_as_uint(t1);
      lo[e] = __float_as_uint(t2);
    }
    pa[s][0] = pack4(hi[0], hi[1], hi[2], hi[3]);
    pa[s][1] = pack4(lo[0], lo[1], lo[2], lo[3]);
    pa[s][2] = pack4(hi[4], hi[5], hi[6], hi[7]);
    pa[s][3] = pack4(lo[4], lo[5], lo[6], lo[7]);
  }

  // PV: n-tile n covers channels 8n .. 8n+7; column g reads channel 8n + g's
  // 16 codes of tokens 16t .. 16t+15 (one 16-byte word, both k-steps).
#pragma unroll
  for (int n = 0; n < 32; ++n) {
    uint4 w = *reinterpret_cast<const uint4*>(rec + kOffVc + (8 * n + g) * kPageTokens + 16 * t);
    int d[4] = {0, 0, 0, 0};
    mma_s8(d, pa[0], w.x, w.y);
    mma_s8(d, pa[1], w.z, w.w);
    float2 u2 = *reinterpret_cast<const float2*>(vs + 8 * n + 2 * t);
    O[n][0] = fmaf(u2.x, (float)(d[0] * 254 + d[2]), O[n][0]);
    O[n][1] = fmaf(u2.y, (float)(d[1] * 254 + d[3]), O[n][1]);
  }
}

// -------------------------------------------------------- BF16 half-page
__device__ __forceinline__ void process_bf16_half(uint8_t* slot, int tok0, int tb, int te, const uint32_t* qrow,
                                                  float qscale, float& m_run, float& l_run, float (&O)[32][2]) {
  const int lane = threadIdx.x & 31, t = lane & 3;
  const uint8_t* K = slot;
  uint8_t* V = slot + 32 * kPad;
  // zero the value rows of tokens outside the range (they may hold anything)
  if (tok0 < tb || tok0 + 32 > te) {
    for (int k = 0; k < 32; ++k) {
      int tok = tok0 + k;
      if (tok < tb || tok >= te) *reinterpret_cast<uint4*>(V + k * kPad + 16 * lane) = make_uint4(0, 0, 0, 0);
    }
    __syncwarp();
  }
  // QK: n-tile j = keys 8j .. 8j+7
  float x[8];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 2
    for (int kk = 0; kk < 8; ++kk) {
      // A: q[g][16 ks + 2t, +1] and q[g][16 ks + 8 + 2t, +1] for k-steps ks = 2kk, 2kk+1
      const uint32_t qa0 = qrow[16 * kk + t], qa1 = qrow[16 * kk + 4 + t];
      const uint32_t qa2 = qrow[16 * kk + 8 + t], qa3 = qrow[16 * kk + 12 + t];
      uint32_t m[4];
      ldsm_x4(m, K + (8 * j + (lane & 7)) * kPad + (4 * kk + (lane >> 3)) * 16);
      mma_bf16(c, qa0, 0u, qa1, 0u, m[0], m[1]);
      mma_bf16(c, qa2, 0u, qa3, 0u, m[2], m[3]);
    }
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      int tok = tok0 + 8 * j + 2 * t + e;
      x[2 * j + e] = (tok >= tb && tok < te) ? c[e] * qscale : kNegInf;
    }
  }
  softmax_update<8>(x, m_run, l_run, O);
  // P as bf16 high/low planes; k-step ks = keys 16 ks .. 16 ks + 15
  uint32_t pa[2][4];
#pragma unroll
  for (int ks = 0; ks < 2; ++ks) {
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      float p0 = x[2 * (2 * ks + hh)], p1 = x[2 * (2 * ks + hh) + 1];
      uint32_t hi = pack_bf16(p0, p1);
      float r0 = p0 - bf16_lo(hi), r1 = p1 - bf16_hi(hi);
      pa[ks][2 * hh] = hi;
      pa[ks][2 * hh + 1] = pack_bf16(r0, r1);
    }
  }
  // PV: pairs of n-tiles (16 channels) per ldmatrix.x4.trans
#pragma unroll
  for (int np = 0; np < 16; ++np) {
    float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
      const int i = lane >> 3;
      uint32_t m[4];
      ldsm_x4_t(m, V + (16 * ks + (i & 1) * 8 + (lane & 7)) * kPad + (2 * np + (i >> 1)) * 16);
      mma_bf16(d0, pa[ks][0], pa[ks][1], pa[ks][2], pa[ks][3], m[0], m[1]);
      mma_bf16(d1, pa[ks][0], pa[ks][1], pa[ks][2], pa[ks][3], m[2], m[3]);
    }
    O[2 * np][0] += d0[0] + d0[2];
    O[2 * np][1] += d0[1] + d0[3];
    O[2 * np + 1][0] += d1[0] + d1[2];
    O[2 * np + 1][1] += d1[1] + d1[3];
  }
}

// ------------------------------------------------------------------ kernel
__global__ void __launch_bounds__(kMmaThreads, 1) decode_mma_kernel(const __grid_constant__ DecodeParams p) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  MmaSmem& S = *reinterpret_cast<MmaSmem*>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t = lane & 3;

  const UnitInfo ui = decode_unit(p, blockIdx.x);
  const Items it = unit_items(ui);
  if (tid == 0) {
    for (int s = 0; s < kMmaSlots; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], 1);
    }
    S.abort = 0;
    fence_mbar_init();
  }
  load_page_table(p, ui, it, S);
  {
    const uint32_t* q32 = reinterpret_cast<const uint32_t*>(p.q + (int64_t)(ui.b * p.H + ui.h) * kGroup * kHeadDim);
    for (int i = tid; i < kGroup * kHeadDim / 2; i += blockDim.x) (&S.q[0][0])[i] = __ldg(q32 + i);
  }
  __syncthreads();

  int issued = 0;
  float O[32][2];
#pragma unroll
  for (int n = 0; n < 32; ++n) O[n][0] = O[n][1] = 0.f;
  float m_run = kNegInf, l_run = 0.f;

  if (warp == kMmaCons) {
    // ---------------------------------------------------------- producer
    if (lane == 0) {
      for (int j = 0; j < it.n; ++j) {
        const int s = j % kMmaSlots;
        if (j >= kMmaSlots && !mbar_wait(&S.empty[s], ((j / kMmaSlots) - 1) & 1, p.status)) {
          S.abort = 1;
          break;
        }
        mma_issue(p, ui, it, S, j, s);
        issued = j + 1;
      }
    }
  } else {
    // ---------------------------------------------------------- consumers
    if (ui.tier == 1) {
      const uint32_t* qrow_s = S.q[g];
      for (int j = warp; j < it.n; j += kMmaCons) {
        const int s = j % kMmaSlots;
        if (!mbar_wait(&S.full[s], (j / kMmaSlots) & 1, p.status)) {
          S.abort = 1;
          break;
        }
        if (S.valid[s]) process_int8_page(S.slot[s], qrow_s, p.qscale, m_run, l_run, O);
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.empty[s]);
      }
    } else {
      const uint32_t* qrow_s = S.q[g];
      for (int j = warp; j < it.n; j += kMmaCons) {
        const int s = j % kMmaSlots;
        if (!mbar_wait(&S.full[s], (j / kMmaSlots) & 1, p.status)) {
          S.abort = 1;
          break;
        }
        if (S.valid[s])
          process_bf16_half(S.slot[s], (it.first + j) * 32, ui.tok_begin, ui.tok_end, qrow_s, p.qscale, m_run,
                            l_run, O);
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.empty[s]);
      }
    }
  }
  __syncthreads();
  if (S.abort) {
    // A wait gave up: let the copies this block issued land (bounded), then leave
    // without a result; the status word reports the timeout.
    if (warp == kMmaCons && lane == 0)
      for (int j = max(0, issued - kMmaSlots); j < issued; ++j)
        mbar_wait(&S.full[j % kMmaSlots], (j / kMmaSlots) & 1, p.status);
    __syncthreads();
    return;
  }
  // ---- per-warp states into shared memory (stages are idle now)
  float* ep_o = reinterpret_cast<float*>(S.slot[0]);
  if (warp < kMmaCons) {
    float L = l_run;
    L += __shfl_xor_sync(kAll, L, 1);
    L += __shfl_xor_sync(kAll, L, 2);
    if (t == 0) {
      S.ep_m[warp][g] = m_run;
      S.ep_l[warp][g] = L;
    }
    const float osc = ui.tier == 1 ? 1.f / (127.f * 254.f) : 1.f;
    float* dst = ep_o + (warp * kGroup + g) * kHeadDim + 2 * t;
#pragma unroll
    for (int n = 0; n < 32; ++n)
      *reinterpret_cast<float2*>(dst + 8 * n) = make_float2(O[n][0] * osc, O[n][1] * osc);
  }
  __syncthreads();
  write_and_fold(p, ui, S, ep_o);
}

cudaError_t launch_decode_mma(const DecodeParams& p, cudaStream_t stream) {
  static bool configured = false;
  const int smem = (int)sizeof(MmaSmem);
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(decode_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  if (p.n_units == 0) return cudaSuccess;
  decode_mma_kernel<<<p.n_units, kMmaThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

int decode_mma_blocks_per_sm() {
  int n = 0;
  const int smem = (int)sizeof(MmaSmem);
  cudaFuncSetAttribute(decode_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_mma_kernel, kMmaThreads, smem) != cudaSuccess)
    return 1;
  return n > 0 ? n : 1;
}

}  // namespace tpk
