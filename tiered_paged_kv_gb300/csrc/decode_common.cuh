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
// On entry each of the NW online-softmax states w (a warp's in the CUDA-core
// kernel, a warp pair's in the tensor-core kernel) is in shared memory for the 8
// query rows: ep_m[w][r] (base-2 running max, integer valued, or -inf),
// ep_l[w][r] (sum of weights) and the unnormalised accumulator in
// ep_o[w][r][RowStride] (shared memory aliasing the idle stages; channels 0..255
// of a row, rows RowStride floats apart).
//
// Threads 0..127 combine the NW states into the unit's partial (o, lse) and
// write it: to the caller's partial arrays (primitive calls), straight to the
// output when the head has a single unit, or to the workspace, where the fold
// kernel merges the head's partials.  Threads 0..127 do the work (row (tid / 16)
// mod 8, 16 channels each); the others return at once.
template <int NW, typename Smem, int RowStride = kHeadDim>
__device__ __forceinline__ void write_and_fold(const DecodeParams& p, const UnitInfo& ui, Smem& S,
                                               const float* ep_o) {
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
        float4 v = *reinterpret_cast<const float4*>(ep_o + (w * G + r) * RowStride + c0 + c);
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
  (void)fold;
}

}  // namespace tpk
