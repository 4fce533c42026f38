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

cudaError_t launch_merge(int n_parts, int rows, const float* o_parts, const float* lse_parts, float* o_acc,
                         float* lse_acc, cudaStream_t stream) {
  if (rows == 0) return cudaSuccess;
  merge_kernel<<<rows, kHeadDim, 0, stream>>>(n_parts, rows, o_parts, lse_parts, o_acc, lse_acc);
  return cudaGetLastError();
}

}  // namespace tpk
