// Lossless 13-bit page format ("model quantization", section "A lossless tier
// first": 13 bits per value, an 18.7 % saving, with a raw fallback when a plane
// needs more than a 32-entry table).
//
// A plane is one page-head's keys (or values), 64 x 256 BF16 values in token-major
// order.  With at most 32 distinct exponent fields, a value is stored as its sign
// and mantissa (one byte) and the 5-bit position of its exponent in the plane's
// ascending exponent table; otherwise the plane is stored raw.  Layouts are in
// tpk.h (TPK_PACK13_*).
//
// Both kernels take one block of 256 threads per page-head and move whole planes
// with 16-byte accesses; thread i of load j handles values 8 (256 j + i) .. + 7, so
// every load and store of a warp is contiguous.  The exponent table needs no
// search: thread e marks exponent e present, and its rank among the present
// exponents (a ballot prefix count) is its table index.
#include <cuda_runtime.h>

#include "common.cuh"

namespace tpk {

constexpr int kP13Threads = 256;
constexpr int kPlaneValues = kPageTokens * kHeadDim;  // 16384
constexpr int kPlaneEnc = 26656;
constexpr int kPlaneRaw = 32768;
constexpr int kP13Header = 16;
constexpr int64_t kP13Record = kP13Header + 2 * kPlaneRaw;
constexpr int kOffSm = 32, kOffLo4 = 32 + 16384, kOffHi1 = 32 + 16384 + 8192;

// sign and mantissa bytes of the two BF16 values in w, at bytes 0 and 2
__device__ __forceinline__ uint32_t sm_pair(uint32_t w) { return ((w >> 8) & 0x00800080u) | (w & 0x007F007Fu); }

__global__ void __launch_bounds__(kP13Threads) pack13_kernel(const __grid_constant__ Pack13Params p) {
  __shared__ uint8_t present[2][256];
  __shared__ uint8_t rank[2][256];
  __shared__ int wcount[2][kP13Threads / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int page = blockIdx.x / p.H, h = blockIdx.x % p.H;
  const int64_t src = p.src[page], dst = p.dst[page];
  if (src < 0 || (p.kv_slots && src >= p.kv_slots) || dst < 0 || (p.out_slots && dst >= p.out_slots)) {
    if (tid == 0) atomicOr(p.status, kStatusBadSlot);
    return;
  }
  const int64_t off = (src * p.H + h) * kPlaneValues;
  const uint4* planes[2] = {reinterpret_cast<const uint4*>(p.k_pool + off),
                            reinterpret_cast<const uint4*>(p.v_pool + off)};
  uint4 x[2][8];
#pragma unroll
  for (int pl = 0; pl < 2; ++pl)
#pragma unroll
    for (int j = 0; j < 8; ++j) x[pl][j] = __ldg(planes[pl] + 256 * j + tid);
  present[0][tid] = 0;
  present[1][tid] = 0;
  __syncthreads();
  // every value marks its exponent field (same-value stores, no atomics needed)
#pragma unroll
  for (int pl = 0; pl < 2; ++pl)
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t w[4] = {x[pl][j].x, x[pl][j].y, x[pl][j].z, x[pl][j].w};
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        present[pl][(w[m] >> 7) & 0xFF] = 1;
        present[pl][(w[m] >> 23) & 0xFF] = 1;
      }
    }
  __syncthreads();
  // thread e: rank of exponent e among the present ones = its table index
  int f[2];
  unsigned bal[2];
#pragma unroll
  for (int pl = 0; pl < 2; ++pl) {
    f[pl] = present[pl][tid];
    bal[pl] = __ballot_sync(0xffffffffu, f[pl]);
    if (lane == 0) wcount[pl][warp] = __popc(bal[pl]);
  }
  __syncthreads();
  int count[2];
#pragma unroll
  for (int pl = 0; pl < 2; ++pl) {
    int below = 0, total = 0;
#pragma unroll
    for (int w = 0; w < kP13Threads / 32; ++w) {
      below += w < warp ? wcount[pl][w] : 0;
      total += wcount[pl][w];
    }
    count[pl] = total;
    rank[pl][tid] = (uint8_t)(below + __popc(bal[pl] & ((1u << lane) - 1u)));
  }
  __syncthreads();
  const int bytes[2] = {count[0] <= 32 ? kPlaneEnc : kPlaneRaw, count[1] <= 32 ? kPlaneEnc : kPlaneRaw};
  uint8_t* rec = p.out + (dst * p.H + h) * kP13Record;
  if (tid == 0) *reinterpret_cast<uint4*>(rec) = make_uint4((unsigned)bytes[0], (unsigned)bytes[1], 0u, 0u);
#pragma unroll
  for (int pl = 0; pl < 2; ++pl) {
    uint8_t* base = rec + kP13Header + (pl ? bytes[0] : 0);
    if (count[pl] > 32) {
#pragma unroll
      for (int j = 0; j < 8; ++j) reinterpret_cast<uint4*>(base)[256 * j + tid] = x[pl][j];
      continue;
    }
    if (f[pl]) base[rank[pl][tid]] = (uint8_t)tid;  // the table, ascending
    if (tid >= count[pl] && tid < 32) base[tid] = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int q = 256 * j + tid;  // values 8q .. 8q + 7
      const uint32_t w[4] = {x[pl][j].x, x[pl][j].y, x[pl][j].z, x[pl][j].w};
      uint32_t nib = 0, hi = 0;
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const uint32_t i0 = rank[pl][(w[m] >> 7) & 0xFF], i1 = rank[pl][(w[m] >> 23) & 0xFF];
        nib |= ((i0 & 15u) << (8 * m)) | ((i1 & 15u) << (8 * m + 4));
        hi |= ((i0 >> 4) << (2 * m)) | ((i1 >> 4) << (2 * m + 1));
      }
      const uint2 sm = make_uint2(__byte_perm(sm_pair(w[0]), sm_pair(w[1]), 0x6420),
                                  __byte_perm(sm_pair(w[2]), sm_pair(w[3]), 0x6420));
      *reinterpret_cast<uint2*>(base + kOffSm + 8 * q) = sm;
      *reinterpret_cast<uint32_t*>(base + kOffLo4 + 4 * q) = nib;
      base[kOffHi1 + q] = (uint8_t)hi;
    }
  }
}

__global__ void __launch_bounds__(kP13Threads) unpack13_kernel(const __grid_constant__ Unpack13Params p) {
  __shared__ uint8_t table[2][32];
  const int tid = threadIdx.x;
  const int page = blockIdx.x / p.H, h = blockIdx.x % p.H;
  const int64_t dst = p.dst[page];
  const int64_t at = p.offsets[blockIdx.x];
  bool ok = dst >= 0 && (p.kv_slots == 0 || dst < p.kv_slots);
  if (!ok) {
    if (tid == 0) atomicOr(p.status, kStatusBadSlot);
    return;
  }
  ok = at >= 0 && (at & 15) == 0 && (p.src_bytes == 0 || at + kP13Header <= p.src_bytes);
  uint4 hdr = make_uint4(0u, 0u, 0u, 0u);
  if (ok) hdr = *reinterpret_cast<const uint4*>(p.src + at);
  const int bytes[2] = {(int)hdr.x, (int)hdr.y};
  ok = ok && (bytes[0] == kPlaneEnc || bytes[0] == kPlaneRaw) && (bytes[1] == kPlaneEnc || bytes[1] == kPlaneRaw) &&
       (p.src_bytes == 0 || at + kP13Header + bytes[0] + bytes[1] <= p.src_bytes);
  if (!ok) {
    if (tid == 0) atomicOr(p.status, kStatusBadRecord);
    return;
  }
  const uint8_t* rec = p.src + at;
  if (tid < 64) {
    const int pl = tid >> 5;
    table[pl][tid & 31] = bytes[pl] == kPlaneEnc ? rec[kP13Header + (pl ? bytes[0] : 0) + (tid & 31)] : 0;
  }
  __syncthreads();
  const int64_t off = (dst * p.H + h) * kPlaneValues;
  uint4* outs[2] = {reinterpret_cast<uint4*>(p.k_pool + off), reinterpret_cast<uint4*>(p.v_pool + off)};
#pragma unroll
  for (int pl = 0; pl < 2; ++pl) {
    const uint8_t* base = rec + kP13Header + (pl ? bytes[0] : 0);
    if (bytes[pl] == kPlaneRaw) {
#pragma unroll
      for (int j = 0; j < 8; ++j) outs[pl][256 * j + tid] = reinterpret_cast<const uint4*>(base)[256 * j + tid];
      continue;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int q = 256 * j + tid;
      const uint2 sm = *reinterpret_cast<const uint2*>(base + kOffSm + 8 * q);
      const uint32_t nib = *reinterpret_cast<const uint32_t*>(base + kOffLo4 + 4 * q);
      const uint32_t hi = base[kOffHi1 + q];
      uint32_t w[4];
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const uint32_t smw = m < 2 ? sm.x : sm.y;
        uint32_t half[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int v = 2 * m + e;  // value 8q + v
          const uint32_t s = (smw >> (8 * (v & 3))) & 0xFFu;
          const uint32_t idx = ((nib >> (4 * v)) & 15u) | (((hi >> v) & 1u) << 4);
          half[e] = ((s & 0x80u) << 8) | ((uint32_t)table[pl][idx] << 7) | (s & 0x7Fu);
        }
        w[m] = half[0] | (half[1] << 16);
      }
      outs[pl][q] = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
}

cudaError_t launch_pack13(const Pack13Params& p, int n_pages, cudaStream_t stream) {
  pack13_kernel<<<n_pages * p.H, kP13Threads, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_unpack13(const Unpack13Params& p, int n_pages, cudaStream_t stream) {
  unpack13_kernel<<<n_pages * p.H, kP13Threads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace tpk
