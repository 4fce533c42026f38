// Log-sum-exp merge of decode partials ("SYCL", section "A merge that joins the
// tiers": one work-group per token and head, one work-item per channel, folding
// the partials of each tier into one FP32 accumulator; -inf is the empty partial).
//
// One thread block per row (query head of the decoded token), one thread per
// channel.  The fold order is fixed: the accumulator, then parts 0, 1, ...
#include "common.cuh"

namespace tpk {

__global__ void __launch_bounds__(kHeadDim) merge_kernel(int n_parts, int rows, const float* __restrict__ o_parts,
                                                         const float* __restrict__ lse_parts, float* o_acc,
                                                         float* lse_acc) {
  const int row = blockIdx.x, c = threadIdx.x;
  const float ninf = -__builtin_huge_valf();
  float la = lse_acc[row];
  float M = la;
  for (int i = 0; i < n_parts; ++i) M = fmaxf(M, lse_parts[(int64_t)i * rows + row]);
  if (M == ninf) return;  // everything empty: the accumulator (0, -inf) stays as it is
  float L = (la == ninf) ? 0.f : expf(la - M);
  for (int i = 0; i < n_parts; ++i) {
    float li = lse_parts[(int64_t)i * rows + row];
    if (li != ninf) L += expf(li - M);
  }
  const float LSE = M + logf(L);
  float acc = (la == ninf) ? 0.f : expf(la - LSE) * o_acc[(int64_t)row * kHeadDim + c];
  for (int i = 0; i < n_parts; ++i) {
    float li = lse_parts[(int64_t)i * rows + row];
    if (li == ninf) continue;
    acc += expf(li - LSE) * o_parts[((int64_t)i * rows + row) * kHeadDim + c];
  }
  __syncthreads();  // every thread has read lse_acc[row] before it is overwritten
  o_acc[(int64_t)row * kHeadDim + c] = acc;
  if (c == 0) lse_acc[row] = LSE;
}

// Fold of the multi-request launch: block (request b, KV head h, row r,
// channel quarter) merges the partials of that head's units, in unit order, for
// 64 channels of one output row; thread c owns one channel.  The lse values are
// staged in shared memory with their merge weights, then every partial's value
// for the thread's channel is loaded in batches of 16 independent loads.
constexpr int kFoldQuarters = 4;
constexpr int kFoldFast = 64;  // heads with at most this many units (= threads per block) fold in one round trip
template <int R>
__global__ void __launch_bounds__(64) fold_kernel(const __grid_constant__ DecodeParams p,
                                                  const __grid_constant__ Plan<R> plan) {
  constexpr int kChunk = 2048;  // partials per shared-memory pass
  __shared__ float lse_s[kChunk];
  __shared__ float w_s[kChunk];
  __shared__ float red_s[2];
  const int G = kGroup;
  const int qtr = blockIdx.x % kFoldQuarters;
  const int row = blockIdx.x / kFoldQuarters;  // (b * H + h) * G + r
  const int b = row / (p.H * G);
  const int h = (row / G) % p.H;
  const int r = row % G;
  const ReqPlan& rp = plan.req[b];
  const int n = rp.splits_e + rp.splits_8;
  if (n <= 1) return;  // a single unit wrote the output itself
  const int first = rp.unit_base + h * n;
  const int c = qtr * 64 + threadIdx.x;
  const float ninf = -__builtin_huge_valf();
  if (n <= kFoldFast) {
    // One memory round trip.  Thread i (< n) owns partial i's lse; the block
    // reduces max and sum with a fixed tree (deterministic), and each thread then
    // combines its channel from values requested right after the wait.
    float v[kFoldFast];
    const float* src = p.part_o + ((int64_t)first * G + r) * kHeadDim + c;
#pragma unroll
    for (int i = 0; i < kFoldFast; ++i) v[i] = i < n ? src[(int64_t)i * G * kHeadDim] : 0.f;
    const int t = threadIdx.x;
    const float li = t < n ? p.part_lse[(first + t) * G + r] : ninf;
    float m = li;
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    if ((t & 31) == 0) red_s[t >> 5] = m;
    __syncthreads();
    const float M = fmaxf(red_s[0], red_s[1]);
    if (M == ninf) {
      p.out_o[(int64_t)row * kHeadDim + c] = 0.f;
      if (c == 0) p.out_lse[row] = ninf;
      return;
    }
    const float wi = (li == ninf) ? 0.f : expf(li - M);
    float sum = wi;
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
    __syncthreads();
    if ((t & 31) == 0) red_s[t >> 5] = sum;
    __syncthreads();
    const float L = red_s[0] + red_s[1];
    if (t < n) w_s[t] = wi / L;
    __syncthreads();
    float acc = 0.f;
#pragma unroll
    for (int i = 0; i < kFoldFast; ++i)
      if (i < n) acc += w_s[i] * v[i];
    p.out_o[(int64_t)row * kHeadDim + c] = acc;
    if (c == 0) p.out_lse[row] = M + logf(L);
    return;
  }
  float M = ninf, L = 0.f;
  for (int i0 = 0; i0 < n; i0 += kChunk) {
    const int cnt = min(kChunk, n - i0);
    __syncthreads();
    for (int i = threadIdx.x; i < cnt; i += blockDim.x) lse_s[i] = p.part_lse[(first + i0 + i) * G + r];
    __syncthreads();
    float bm = ninf;
    for (int i = 0; i < cnt; ++i) bm = fmaxf(bm, lse_s[i]);
    if (bm == ninf) continue;
    if (bm > M) {
      L = (M == ninf) ? 0.f : L * expf(M - bm);
      M = bm;
    }
    for (int i = 0; i < cnt; ++i)
      if (lse_s[i] != ninf) L += expf(lse_s[i] - M);
  }
  if (M == ninf) {
    p.out_o[(int64_t)row * kHeadDim + c] = 0.f;
    if (c == 0) p.out_lse[row] = ninf;
    return;
  }
  const float LSE = M + logf(L);
  float acc = 0.f;
  for (int i0 = 0; i0 < n; i0 += kChunk) {
    const int cnt = min(kChunk, n - i0);
    __syncthreads();
    for (int i = threadIdx.x; i < cnt; i += blockDim.x) {
      const float li = p.part_lse[(first + i0 + i) * G + r];
      w_s[i] = (li == ninf) ? 0.f : expf(li - LSE);
    }
    __syncthreads();
    const float* src = p.part_o + ((int64_t)(first + i0) * G + r) * kHeadDim + c;
    for (int j0 = 0; j0 < cnt; j0 += 16) {
      float v[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) v[k] = (j0 + k < cnt) ? src[(int64_t)(j0 + k) * G * kHeadDim] : 0.f;
#pragma unroll
      for (int k = 0; k < 16; ++k)
        if (j0 + k < cnt && w_s[j0 + k] != 0.f) acc += w_s[j0 + k] * v[k];
    }
  }
  p.out_o[(int64_t)row * kHeadDim + c] = acc;
  if (c == 0) p.out_lse[row] = LSE;
}

template <int R>
static cudaError_t launch_fold_t(const DecodeParams& p, const ReqPlan* req, cudaStream_t stream) {
  Plan<R> plan = {};
  for (int b = 0; b < p.n_req; ++b) plan.req[b] = req[b];
  fold_kernel<R><<<p.n_req * p.H * kGroup * kFoldQuarters, 64, 0, stream>>>(p, plan);
  return cudaGetLastError();
}

cudaError_t launch_fold(const DecodeParams& p, const ReqPlan* req, cudaStream_t stream) {
  return p.n_req <= kShortPlan ? launch_fold_t<kShortPlan>(p, req, stream)
                               : launch_fold_t<kMaxReqPerLaunch>(p, req, stream);
}

cudaError_t launch_merge(int n_parts, int rows, const float* o_parts, const float* lse_parts, float* o_acc,
                         float* lse_acc, cudaStream_t stream) {
  if (rows == 0) return cudaSuccess;
  merge_kernel<<<rows, kHeadDim, 0, stream>>>(n_parts, rows, o_parts, lse_parts, o_acc, lse_acc);
  return cudaGetLastError();
}

}  // namespace tpk
