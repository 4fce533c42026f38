// Split-tier paged decode attention, CUDA-core (SIMT) dot products.
//
// One thread block = one unit: a contiguous range of pages of one tier for one
// (request, KV head).  Thread 0 streams the unit's items (BF16 half-pages or
// 8-bit records) into a ring of shared-memory stages with 1-D bulk copies
// (cp.async.bulk + mbarrier).  Each of the 4 warps takes a quarter of every
// item's tokens and keeps its own online-softmax state for the 8 query rows of
// the GQA group; lane l owns channels 8l .. 8l+7 of the query rows and of the
// output accumulator.  The epilogue combines the warps and writes the unit's
// partial (o, lse), and in fold mode the last unit of a (request, head) merges
// that head's partials.
//
// Method (pages by title):
//   "SYCL", "Attention that reads 8-bit history": the per-token key factor r_t is
//     applied after the dot product; values are scaled per channel per page.
//   "SYCL", "Exact tricks and a two-owner decoder": the running maximum is kept as
//     an integer in base 2, so every rescale factor is a power of two built by
//     exponent arithmetic, and the rescale is skipped when all eight rows'
//     factors are exactly 1 (a warp vote).
//   "SYCL", "A merge that joins the tiers": log-sum-exp partials.
#include "decode_common.cuh"

namespace tpk {

constexpr unsigned kFull = 0xffffffffu;

// Sum a 32-entry per-lane vector over the warp; afterwards lane l holds the
// total of entry l (a butterfly that halves the vector at every step).
__device__ __forceinline__ float reduce_scatter32(float (&v)[32]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) {
    const bool upper = lane & m;
#pragma unroll
    for (int i = 0; i < m; ++i) {
      float send = upper ? v[i] : v[i + m];
      float keep = upper ? v[i + m] : v[i];
      v[i] = keep + __shfl_xor_sync(kFull, send, m);
    }
  }
  return v[0];
}

// 8 stored code bytes (two words) -> the codes as floats, exactly: each byte
// (the code plus 128) is placed in the mantissa of 2^23 and 2^23 + 128 is subtracted.
__device__ __forceinline__ void codes8_to_float(uint2 w, float (&f)[8]) {
  const uint32_t a = w.x, b = w.y;
  const float bias = 8388736.0f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[i] = __uint_as_float(__byte_perm(a, 0x4b000000u, 0x7540 | i)) - bias;
    f[4 + i] = __uint_as_float(__byte_perm(b, 0x4b000000u, 0x7540 | i)) - bias;
  }
}

__device__ __forceinline__ void bf16x8_to_float(uint4 w, float (&f)[8]) {
  f[0] = bf16_lo(w.x);
  f[1] = bf16_hi(w.x);
  f[2] = bf16_lo(w.y);
  f[3] = bf16_hi(w.y);
  f[4] = bf16_lo(w.z);
  f[5] = bf16_hi(w.z);
  f[6] = bf16_lo(w.w);
  f[7] = bf16_hi(w.w);
}

// The 8-bit record stores value codes channel-major ([256][64]); the CUDA-core
// path reads them token-major, so the block transposes them in place once the
// record has landed (each thread moves a 4-channel x 32-token block, with 4x4
// byte transposes in registers).
__device__ __forceinline__ void transpose_value_codes(uint8_t* vc) {
  const int a = threadIdx.x & 63, b = threadIdx.x >> 6;
  uint32_t w[4][8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint4* src = reinterpret_cast<const uint4*>(vc + vc_byte(4 * a + i, 32 * b));
    uint4 x = src[0], y = src[1];
    w[i][0] = x.x; w[i][1] = x.y; w[i][2] = x.z; w[i][3] = x.w;
    w[i][4] = y.x; w[i][5] = y.y; w[i][6] = y.z; w[i][7] = y.w;
  }
  __syncthreads();
#pragma unroll
  for (int kw = 0; kw < 8; ++kw) {
    uint32_t t01lo = __byte_perm(w[0][kw], w[1][kw], 0x5140), t01hi = __byte_perm(w[0][kw], w[1][kw], 0x7362);
    uint32_t t23lo = __byte_perm(w[2][kw], w[3][kw], 0x5140), t23hi = __byte_perm(w[2][kw], w[3][kw], 0x7362);
    uint32_t o[4] = {__byte_perm(t01lo, t23lo, 0x5410), __byte_perm(t01lo, t23lo, 0x7632),
                     __byte_perm(t01hi, t23hi, 0x5410), __byte_perm(t01hi, t23hi, 0x7632)};
#pragma unroll
    for (int e = 0; e < 4; ++e)
      *reinterpret_cast<uint32_t*>(vc + (32 * b + 4 * kw + e) * kHeadDim + 4 * a) = o[e];
  }
  __syncthreads();
}

// Online-softmax state of one warp.
struct SoftmaxState {
  float m_run;   // base-2 running max of row (lane & 7), integer valued (or -inf)
  float l_lane;  // sum of weights for (key slot lane >> 3, row lane & 7)
};

// One batch of 4 keys: x = score (base 2) of (key lane >> 3, row lane & 7), -inf
// if masked.  Updates the state, rescales O when any row's maximum moved, and
// returns the weight p of (key, row).
__device__ __forceinline__ float softmax_step(SoftmaxState& st, float x, float (&O)[kGroup][8]) {
  float bm = x;
  bm = fmaxf(bm, __shfl_xor_sync(kFull, bm, 8));
  bm = fmaxf(bm, __shfl_xor_sync(kFull, bm, 16));
  float m_new = (bm == kNegInf) ? st.m_run : fmaxf(st.m_run, ceilf(bm));
  float alpha = (m_new == st.m_run) ? 1.f : (st.m_run == kNegInf ? 0.f : ldexpf(1.f, (int)(st.m_run - m_new)));
  float p = (x == kNegInf) ? 0.f : exp2f(x - m_new);
  st.l_lane = st.l_lane * alpha + p;
  st.m_run = m_new;
  // eight-row vote: skip the rescale when every row's factor is exactly 1
  if (!__all_sync(kFull, alpha == 1.f)) {
#pragma unroll
    for (int r = 0; r < kGroup; ++r) {
      float a = __shfl_sync(kFull, alpha, r);
#pragma unroll
      for (int c = 0; c < 8; ++c) O[r][c] *= a;
    }
  }
  return p;
}

template <int R>
__global__ void __launch_bounds__(kDecThreads, 2) decode_simt_kernel(const __grid_constant__ DecodeParams p,
                                                                   const __grid_constant__ Plan<R> plan) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  DecSmem& S = *reinterpret_cast<DecSmem*>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  const UnitInfo ui = decode_unit(p, plan.req, blockIdx.x);
  const Items it = unit_items(ui);

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(&S.full[s], 1);
    fence_mbar_init();
  }
  load_page_table(p, ui, it, S);
  __syncthreads();
  if (tid == 0)
    for (int j = 0; j < min(kStages, it.n); ++j) issue_item(p, ui, it, S, j, j);

  // query rows of this (request, head), pre-scaled to base-2 score units
  float qf[kGroup][8];
  {
    const uint16_t* q = p.q + ((int64_t)(ui.b * p.H + ui.h) * kGroup) * kHeadDim + lane * 8;
#pragma unroll
    for (int r = 0; r < kGroup; ++r) {
      uint4 w = __ldg(reinterpret_cast<const uint4*>(q + r * kHeadDim));
      bf16x8_to_float(w, qf[r]);
#pragma unroll
      for (int c = 0; c < 8; ++c) qf[r][c] *= p.qscale;
    }
  }
  float O[kGroup][8];
#pragma unroll
  for (int r = 0; r < kGroup; ++r)
#pragma unroll
    for (int c = 0; c < 8; ++c) O[r][c] = 0.f;
  SoftmaxState st{kNegInf, 0.f};
  int stop = -1;  // item at which a bounded wait gave up

  for (int j = 0; j < it.n; ++j) {
    const int s = j % kStages;
    const bool landed = mbar_wait(&S.full[s], (j / kStages) & 1, p.status, p.wait_ns);
    if (!__syncthreads_and(landed)) {  // the block agrees on whether a wait gave up
      stop = j;
      break;
    }
    if (S.valid[s]) {
      uint8_t* slot = S.slot[s];
      if (ui.tier == 1) transpose_value_codes(slot + kOffVc);
      if (ui.tier == 0) {
        // ---------------- exact tier: 32 BF16 tokens, 8 per warp
        const uint16_t* Ks = reinterpret_cast<const uint16_t*>(slot);
        const uint16_t* Vs = Ks + 32 * kHeadDim;
        const int tok0 = (it.first + j) * 32;
#pragma unroll 1
        for (int bb = 0; bb < 2; ++bb) {
          const int key0 = warp * 8 + bb * 4;
          float acc[32];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int tok = tok0 + key0 + i;
            const bool ok = tok >= ui.tok_begin && tok < ui.tok_end;
            float k[8];
            if (ok) {
              bf16x8_to_float(*reinterpret_cast<const uint4*>(Ks + (key0 + i) * kHeadDim + lane * 8), k);
            } else {
#pragma unroll
              for (int c = 0; c < 8; ++c) k[c] = 0.f;
            }
#pragma unroll
            for (int r = 0; r < kGroup; ++r) {
              float a = 0.f;
#pragma unroll
              for (int c = 0; c < 8; ++c) a = fmaf(qf[r][c], k[c], a);
              acc[i * 8 + r] = a;
            }
          }
          float x = reduce_scatter32(acc);
          const int mytok = tok0 + key0 + (lane >> 3);
          if (mytok < ui.tok_begin || mytok >= ui.tok_end) x = kNegInf;
          float pw = softmax_step(st, x, O);
          S.pbuf[warp][lane] = pw;
          __syncwarp();
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int tok = tok0 + key0 + i;
            if (tok < ui.tok_begin || tok >= ui.tok_end) continue;
            float v[8];
            bf16x8_to_float(*reinterpret_cast<const uint4*>(Vs + (key0 + i) * kHeadDim + lane * 8), v);
            float4 p0 = *reinterpret_cast<const float4*>(&S.pbuf[warp][i * 8]);
            float4 p1 = *reinterpret_cast<const float4*>(&S.pbuf[warp][i * 8 + 4]);
            float pr[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
#pragma unroll
            for (int r = 0; r < kGroup; ++r)
#pragma unroll
              for (int c = 0; c < 8; ++c) O[r][c] = fmaf(pr[r], v[c], O[r][c]);
          }
          __syncwarp();
        }
      } else {
        // ---------------- 8-bit tier: one 64-token record, 16 tokens per warp
        const uint8_t* kc = slot + kOffKc;
        const uint8_t* vc = slot + kOffVc;  // token-major after the transpose
        const float* ks = reinterpret_cast<const float*>(slot + kOffKsChan);
        const float* kr = reinterpret_cast<const float*>(slot + kOffKsTok);
        const float* vs = reinterpret_cast<const float*>(slot + kOffVsChan);
        float sc[8], uc[8];
        {
          float4 a = *reinterpret_cast<const float4*>(ks + ks_index(lane * 8));
          float4 b = *reinterpret_cast<const float4*>(ks + ks_index(lane * 8 + 4));
          float4 c = *reinterpret_cast<const float4*>(vs + lane * 8);
          float4 d = *reinterpret_cast<const float4*>(vs + lane * 8 + 4);
          sc[0] = a.x; sc[1] = a.y; sc[2] = a.z; sc[3] = a.w;
          sc[4] = b.x; sc[5] = b.y; sc[6] = b.z; sc[7] = b.w;
          uc[0] = c.x; uc[1] = c.y; uc[2] = c.z; uc[3] = c.w;
          uc[4] = d.x; uc[5] = d.y; uc[6] = d.z; uc[7] = d.w;
        }
        const int tok0 = (it.first + j) * kPageTokens;
#pragma unroll 1
        for (int bb = 0; bb < 4; ++bb) {
          const int key0 = warp * 16 + bb * 4;
          float acc[32];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            float k[8];
            codes8_to_float(*reinterpret_cast<const uint2*>(kc + kc_byte(key0 + i, lane * 8)), k);
#pragma unroll
            for (int c = 0; c < 8; ++c) k[c] *= sc[c];
#pragma unroll
            for (int r = 0; r < kGroup; ++r) {
              float a = 0.f;
#pragma unroll
              for (int c = 0; c < 8; ++c) a = fmaf(qf[r][c], k[c], a);
              acc[i * 8 + r] = a;
            }
          }
          float x = reduce_scatter32(acc) * kr[key0 + (lane >> 3)];
          const int mytok = tok0 + key0 + (lane >> 3);
          if (mytok < ui.tok_begin || mytok >= ui.tok_end) x = kNegInf;
          float pw = softmax_step(st, x, O);
          S.pbuf[warp][lane] = pw;
          __syncwarp();
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            float v[8];
            codes8_to_float(*reinterpret_cast<const uint2*>(vc + (key0 + i) * kHeadDim + lane * 8), v);
            float4 p0 = *reinterpret_cast<const float4*>(&S.pbuf[warp][i * 8]);
            float4 p1 = *reinterpret_cast<const float4*>(&S.pbuf[warp][i * 8 + 4]);
            float pr[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
#pragma unroll
            for (int c = 0; c < 8; ++c) v[c] *= uc[c];
#pragma unroll
            for (int r = 0; r < kGroup; ++r)
#pragma unroll
              for (int c = 0; c < 8; ++c) O[r][c] = fmaf(pr[r], v[c], O[r][c]);
          }
          __syncwarp();
        }
      }
    }
    __syncthreads();  // every warp is done with stage s
    if (tid == 0 && j + kStages < it.n) issue_item(p, ui, it, S, j + kStages, s);
  }

  if (stop >= 0) {
    // A copy did not land in time: let the stages still in flight land (bounded)
    // and leave without writing a result; the status word reports the timeout.
    if (tid == 0)
      for (int jj = stop; jj < min(stop + kStages, it.n); ++jj)
        mbar_wait(&S.full[jj % kStages], (jj / kStages) & 1, p.status, p.wait_ns);
    __syncthreads();
    return;
  }

  // ---- epilogue: per-warp row sums and accumulators into shared memory
  float L = st.l_lane;
  L += __shfl_xor_sync(kFull, L, 8);
  L += __shfl_xor_sync(kFull, L, 16);
  if (lane < kGroup) {
    S.ep_m[warp][lane] = st.m_run;
    S.ep_l[warp][lane] = L;
  }
  float* ep_o = reinterpret_cast<float*>(S.slot[0]);  // [warp][row][256], stages are idle now
#pragma unroll
  for (int r = 0; r < kGroup; ++r) {
    float* dst = ep_o + (warp * kGroup + r) * kHeadDim + lane * 8;
    *reinterpret_cast<float4*>(dst) = make_float4(O[r][0], O[r][1], O[r][2], O[r][3]);
    *reinterpret_cast<float4*>(dst + 4) = make_float4(O[r][4], O[r][5], O[r][6], O[r][7]);
  }
  __syncthreads();
  write_and_fold<kDecWarps>(p, ui, S, ep_o);
}

template <int R>
static cudaError_t launch_simt(const DecodeParams& p, const ReqPlan* req, cudaStream_t stream) {
  static DeviceOnce once;
  const int smem = (int)sizeof(DecSmem);
  cudaError_t e = once.run(
      [&] { return cudaFuncSetAttribute(decode_simt_kernel<R>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem); });
  if (e != cudaSuccess) return e;
  Plan<R> plan = {};
  for (int b = 0; b < p.n_req; ++b) plan.req[b] = req[b];
  decode_simt_kernel<R><<<p.n_units, kDecThreads, smem, stream>>>(p, plan);
  return cudaGetLastError();
}

cudaError_t launch_decode_simt(const DecodeParams& p, const ReqPlan* req, cudaStream_t stream) {
  if (p.n_units == 0) return cudaSuccess;
  return p.n_req <= kShortPlan ? launch_simt<kShortPlan>(p, req, stream)
                               : launch_simt<kMaxReqPerLaunch>(p, req, stream);
}

int decode_simt_blocks_per_sm() {
  int n = 0;
  const int smem = (int)sizeof(DecSmem);
  cudaFuncSetAttribute(decode_simt_kernel<kMaxReqPerLaunch>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_simt_kernel<kMaxReqPerLaunch>, kDecThreads, smem) !=
      cudaSuccess)
    return 1;
  return n > 0 ? n : 1;
}

}  // namespace tpk
