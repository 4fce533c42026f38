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

// Fold of the multi-request launch: block (request b, KV head h, row r) merges
// the partials of that head's units, in unit order, for one output row; thread c
// owns channel c.  All the lse values are staged in shared memory first and the
// o loads are issued in batches, so the fold costs a few memory round trips.
__global__ void __launch_bounds__(kHeadDim) fold_kernel(const __grid_constant__ DecodeParams p) {
  __shared__ float lse_s[1024];
  __shared__ float w_s[1024];
  const int G = kGroup;
  const int b = blockIdx.x / (p.H * G);
  const int h = (blockIdx.x / G) % p.H;
  const int r = blockIdx.x % G;
  const ReqPlan& rp = p.req[b];
  const int n = rp.splits_e + rp.splits_8;
  if (n <= 1) return;  // a single unit wrote the output itself
  const int first = rp.unit_base + h * n;
  const int c = threadIdx.x;
  const float ninf = -__builtin_huge_valf();
  const int row_out = (b * p.H + h) * G + r;
  float M = ninf, L = 0.f;
  for (int i0 = 0; i0 < n; i0 += 1024) {
    const int cnt = min(1024, n - i0);
    __syncthreads();
    for (int i = c; i < cnt; i += blockDim.x) lse_s[i] = p.part_lse[(first + i0 + i) * G + r];
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
    p.out_o[(int64_t)row_out * kHeadDim + c] = 0.f;
    if (c == 0) p.out_lse[row_out] = ninf;
    return;
  }
  const float LSE = M + logf(L);
  float acc = 0.f;
  for (int i0 = 0; i0 < n; i0 += 1024) {
    const int cnt = min(1024, n - i0);
    __syncthreads();
    for (int i = c; i < cnt; i += blockDim.x) {
      const float li = p.part_lse[(first + i0 + i) * G + r];
      w_s[i] = (li == ninf) ? 0.f : expf(li - LSE);
    }
    __syncthreads();
    const float* src = p.part_o + ((int64_t)(first + i0) * G + r) * kHeadDim + c;
    int i = 0;
    for (; i + 8 <= cnt; i += 8) {
      float v[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) v[k] = src[(int64_t)(i + k) * G * kHeadDim];
#pragma unroll
      for (int k = 0; k < 8; ++k)
        if (w_s[i + k] != 0.f) acc += w_s[i + k] * v[k];
    }
    for (; i < cnt; ++i)
      if (w_s[i] != 0.f) acc += w_s[i] * src[(int64_t)i * G * kHeadDim];
  }
  p.out_o[(int64_t)row_out * kHeadDim + c] = acc;
  if (c == 0) p.out_lse[row_out] = LSE;
}

cudaError_t launch_fold(const DecodeParams& p, cudaStream_t stream) {
  fold_kernel<<<p.n_req * p.H * kGroup, kHeadDim, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_merge(int n_parts, int rows, const float* o_parts, const float* lse_parts, float* o_acc,
                         float* lse_acc, cudaStream_t stream) {
  if (rows == 0) return cudaSuccess;
  merge_kernel<<<rows, kHeadDim, 0, stream>>>(n_parts, rows, o_parts, lse_parts, o_acc, lse_acc);
  return cudaGetLastError();
}

}  // namespace tpk
