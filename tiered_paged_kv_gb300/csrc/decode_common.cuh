// Pieces shared by the decode kernels: the shared-memory stage ring fed by bulk
// copies, the per-unit item schedule, and the epilogue that turns per-warp
// online-softmax states into a partial (o, lse) and folds the partials of one
// (request, KV head) in a fixed order.
#pragma once
#include "common.cuh"

namespace tpk {

constexpr int kDecWarps = 4;
constexpr int kDecThreads = kDecWarps * 32;
constexpr int kStages = 3;
constexpr int kSlotBytes = kRecordBytes;  // one 8-bit record, or a BF16 half-page (K 16 KB + V 16 KB)
constexpr int kPtCache = 1024;            // page-table entries staged in shared memory
constexpr float kNegInf = -__builtin_huge_valf();

struct DecSmem {
  alignas(128) uint8_t slot[kStages][kSlotBytes];
  uint64_t full[kStages];
  int valid[kStages];
  int pt[kPtCache];
  alignas(16) float pbuf[kDecWarps][32];
  float ep_m[kDecWarps][kGroup];
  float ep_l[kDecWarps][kGroup];
  int is_last;
};

// Items of a unit: BF16 half-pages (32 tokens) for the exact tier, whole pages
// (64 tokens) for the 8-bit tier.
struct Items {
  int n;         // number of items
  int first;     // exact tier: first half-page index; 8-bit tier: first page index
  int pg_first;  // first page index covered
  int n_pages;   // pages covered
};

__device__ __forceinline__ Items unit_items(const UnitInfo& ui) {
  Items it;
  if (ui.tok_end <= ui.tok_begin) {
    it.n = 0;
    it.first = 0;
    it.pg_first = 0;
    it.n_pages = 0;
  } else if (ui.tier == 0) {
    it.first = ui.tok_begin >> 5;
    it.n = ((ui.tok_end + 31) >> 5) - it.first;
    it.pg_first = ui.tok_begin >> 6;
    it.n_pages = ((ui.tok_end + 63) >> 6) - it.pg_first;
  } else {
    it.first = ui.tok_begin >> 6;
    it.n = (ui.tok_end - ui.tok_begin) >> 6;
    it.pg_first = it.first;
    it.n_pages = it.n;
  }
  return it;
}

__device__ __forceinline__ int item_page(const UnitInfo& ui, const Items& it, int j) {
  return ui.tier == 0 ? (it.first + j) >> 1 : it.first + j;
}

// Stage the unit's page-table entries (first kPtCache of them).
template <typename Smem>
__device__ __forceinline__ void load_page_table(const DecodeParams& p, const UnitInfo& ui, const Items& it,
                                                Smem& S) {
  const int32_t* pt = (ui.tier == 0 ? p.page_table : p.page_table8) + ui.pt_off + it.pg_first;
  int n = min(it.n_pages, kPtCache);
  for (int i = threadIdx.x; i < n; i += blockDim.x) S.pt[i] = __ldg(pt + i);
}

// Issue the bulk copy of item j into stage s (called by one thread).  An entry
// outside the pool is not read: the stage is marked invalid and its barrier is
// completed without a transfer.
__device__ __forceinline__ void issue_item(const DecodeParams& p, const UnitInfo& ui, const Items& it,
                                           DecSmem& S, int j, int s) {
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
    int half = (it.first + j) & 1;
    int64_t off = ((slot * p.H + ui.h) * kPageTokens + half * 32) * (int64_t)kHeadDim;
    mbar_arrive_expect_tx(&S.full[s], 32768);
    bulk_g2s(S.slot[s], p.k_pool + off, 16384, &S.full[s]);
    bulk_g2s(S.slot[s] + 16384, p.v_pool + off, 16384, &S.full[s]);
  } else {
    const uint8_t* src = p.rec_pool + (slot * p.H + ui.h) * (int64_t)kRecordBytes;
    mbar_arrive_expect_tx(&S.full[s], kRecordBytes);
    bulk_g2s(S.slot[s], src, kRecordBytes, &S.full[s]);
  }
}

// -------------------------------------------------------------- epilogue
// On entry every one of the NW consumer warps w has stored its online-softmax state for the 8
// query rows: ep_m[w][r] (base-2 running max, integer valued, or -inf),
// ep_l[w][r] (sum of weights) and its unnormalised accumulator in
// ep_o[w][r][256] (shared memory aliasing the idle stages).
//
// Threads 0..127 combine the NW warps into the unit's partial (o, lse)
// and write it; in fold mode the last unit of a (request, KV head) then merges
// all of that head's partials in unit order (a fixed order, so the result does
// not depend on which unit finished last).  `scratch` is idle shared memory.  Every thread of the block must
// call this (it contains block barriers); threads >= 128 only take part in them.
template <int NW, typename Smem>
__device__ __forceinline__ void write_and_fold(const DecodeParams& p, const UnitInfo& ui, Smem& S,
                                               const float* ep_o, float* scratch, int scratch_floats) {
  const int tid = threadIdx.x;
  const bool worker = tid < 128;
  const int G = kGroup;
  float* dst_o;
  float* dst_lse;
  bool fold = false;
  const int row0_final = (ui.b * p.H + ui.h) * G;
  if (p.mode == kModePrimitive) {
    int row0 = (ui.split * p.H + ui.h) * G;
    dst_o = p.part_o + (int64_t)row0 * kHeadDim;
    dst_lse = p.part_lse + row0;
  } else if (ui.per_head == 1) {
    dst_o = p.out_o + (int64_t)row0_final * kHeadDim;
    dst_lse = p.out_lse + row0_final;
  } else {
    dst_o = p.part_o + (int64_t)blockIdx.x * G * kHeadDim;
    dst_lse = p.part_lse + blockIdx.x * G;
    fold = true;
  }
  const int r = (tid >> 4) & 7;
  const int c0 = (tid & 15) * 16;
  if (worker) {
    float M = kNegInf;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, S.ep_m[w][r]);
    float fw[NW];
    float L = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      float mw = S.ep_m[w][r];
      fw[w] = (mw == kNegInf) ? 0.f : ldexpf(1.f, (int)(mw - M));
      L += fw[w] * S.ep_l[w][r];
    }
    const bool empty = !(L > 0.f);
    const float inv = empty ? 0.f : 1.f / L;
#pragma unroll
    for (int c = 0; c < 16; c += 4) {
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        float4 v = *reinterpret_cast<const float4*>(ep_o + (w * G + r) * kHeadDim + c0 + c);
        acc.x += fw[w] * v.x;
        acc.y += fw[w] * v.y;
        acc.z += fw[w] * v.z;
        acc.w += fw[w] * v.w;
      }
      acc.x *= inv;
      acc.y *= inv;
      acc.z *= inv;
      acc.w *= inv;
      *reinterpret_cast<float4*>(dst_o + r * kHeadDim + c0 + c) = acc;
    }
    if ((tid & 15) == 0) dst_lse[r] = empty ? kNegInf : (M + log2f(L)) * kLn2;
  }
  if (!fold) return;
  // ---- fold: the last unit of this (request, head) merges all its partials
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    int* ticket = p.tickets + ui.b * p.H + ui.h;
    int prev = atomicAdd(ticket, 1);
    S.is_last = (prev == ui.per_head - 1);
    if (S.is_last) *ticket = 0;  // leave the workspace zeroed for the next launch
  }
  __syncthreads();
  if (!S.is_last) return;
  __threadfence();
  const int first = blockIdx.x - ui.unit_in_head;
  const int n = ui.per_head;
  // stage the head's partial lse values [n][8] in shared memory (they are
  // contiguous in the workspace), using the idle stage memory as scratch
  float* lse_s = scratch;
  const bool staged = n * G <= scratch_floats;
  if (staged)
    for (int i = tid; i < n * G; i += blockDim.x) lse_s[i] = __ldcg(p.part_lse + first * G + i);
  __syncthreads();
  if (!worker) return;
  auto lse_at = [&](int i) { return staged ? lse_s[i * G + r] : __ldcg(p.part_lse + (first + i) * G + r); };
  float M = kNegInf;
  for (int i = 0; i < n; ++i) M = fmaxf(M, lse_at(i));
  float* out_o = p.out_o + (int64_t)(row0_final + r) * kHeadDim + c0;
  if (M == kNegInf) {
#pragma unroll
    for (int c = 0; c < 16; ++c) out_o[c] = 0.f;
    if ((tid & 15) == 0) p.out_lse[row0_final + r] = kNegInf;
    return;
  }
  float L = 0.f;
  for (int i = 0; i < n; ++i) {
    float li = lse_at(i);
    if (li != kNegInf) L += expf(li - M);
  }
  const float LSE = M + logf(L);
  float acc[16];
#pragma unroll
  for (int c = 0; c < 16; ++c) acc[c] = 0.f;
  // four partials per iteration keep 16 independent 16-byte loads in flight
  for (int i0 = 0; i0 < n; i0 += 4) {
    float4 v[4][4];
    float wgt[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int i = i0 + k;
      const float li = i < n ? lse_at(i) : kNegInf;
      wgt[k] = (li == kNegInf) ? 0.f : expf(li - LSE);
      const float4* src =
          reinterpret_cast<const float4*>(p.part_o + ((int64_t)(first + min(i, n - 1)) * G + r) * kHeadDim + c0);
#pragma unroll
      for (int c = 0; c < 4; ++c) v[k][c] = (wgt[k] != 0.f) ? __ldcg(src + c) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int k = 0; k < 4; ++k)
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        acc[4 * c + 0] += wgt[k] * v[k][c].x;
        acc[4 * c + 1] += wgt[k] * v[k][c].y;
        acc[4 * c + 2] += wgt[k] * v[k][c].z;
        acc[4 * c + 3] += wgt[k] * v[k][c].w;
      }
  }
#pragma unroll
  for (int c = 0; c < 16; c += 4)
    *reinterpret_cast<float4*>(out_o + c) = make_float4(acc[c], acc[c + 1], acc[c + 2], acc[c + 3]);
  if ((tid & 15) == 0) p.out_lse[row0_final + r] = LSE;
}

}  // namespace tpk
