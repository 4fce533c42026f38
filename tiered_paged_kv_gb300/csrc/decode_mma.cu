// Split-tier paged decode attention on the tensor cores (mma.sync, f16/bf16 with
// FP32 accumulation).
//
// One thread block = one unit (a range of pages of one tier for one (request,
// KV head)).  The unit's items stream into a ring of 6 shared-memory slots: the
// first three are issued at the start, the next three after the prologue, and
// every later one by the warp that lets go of its slot's previous item last.  8 warps work in 4 pairs: item j goes to
// pair j % 4, and the two warps of the pair split the item's channels in halves
// (partial scores are summed through shared memory, both warps run the same
// online softmax, each accumulates the output of its 128 channels).  The
// epilogue merges the 4 pairs' states.
//
// Thread (g, t) = (lane / 4, lane % 4) of a warp:
//   - in QK (S = Q K^T, M = 16 query-row slots, N = 8 tokens per tile) it owns
//     query row g and receives the scores of 2 tokens per tile;
//   - in PV the output is computed transposed, O^T = V^T P^T (M = 16 channels,
//     N = 8 query rows, K = tokens), so the accumulator is exactly the output:
//     thread (g, t) holds channels 16m + g and 16m + g + 8 of rows 2t, 2t + 1.
//
// 8-bit tier ("SYCL", "Attention that reads 8-bit history").  The codes are exact
// in f16, so both products run on f16 tensor cores:
//   QK  A = the folded query q'_c = q_c s_c, split into f16 high and low planes
//         (rows 0-7 and 8-15 of the tile), B = key codes; the per-token factor r_t
//         is applied to the scores after the dot product;
//   PV  A = value codes (channel-major, so four consecutive tokens of a channel
//         are one word), B = the probabilities as one f16 plane (the weights are
//         rounded to f16 before they enter the row sums too); each page's result
//         is rescaled by its value scale u_c and added to the FP32 accumulator --
//         PV runs on raw codes and is rescaled per page.
// The stored code bytes (code + 128) widen to f16 as 1152 + code with one byte
// permute per two codes; the 1152 offset is removed once per page and row: from
// the scores as 1152 * sum_c q'_c, and from the PV accumulator, which starts at
// -1152 * sum_t p_t.
// The integer tensor path runs at about a quarter of the f16 rate on this GPU, so
// the default keeps the query in floating point; the integer-query variant (the
// pages' "integer query cache") runs QK on it with the operands swapped so that
// no row of the tile is idle (qk_int_query below).
//
// Exact tier: BF16 half-pages (32 tokens) arrive by TMA tensor copies in the
// 128-byte-swizzled layout, so ldmatrix reads are conflict-free; q is exact in
// bf16; P enters as bf16 high and low planes.
//
// Online softmax ("SYCL", "Exact tricks and a two-owner decoder"): the running
// maximum is an integer in base 2, every rescale is a power of two built by
// exponent arithmetic, and the rescale is skipped when no row's maximum moved
// (a warp vote).
#include <cuda_fp16.h>

#include "decode_common.cuh"

namespace tpk {

constexpr int kCons = 8;  // warps (4 pairs), all of them consumers
constexpr int kMmaThreads = kCons * 32;
constexpr int kMmaSlots = 6;
constexpr int kFirstIssue = 3;  // items issued before the prologue
constexpr unsigned kAll = 0xffffffffu;

// float query rows padded by 64 bytes, so that rows g and g + 1 sit in opposite
// bank halves for the contiguous row reads of the integer-query absmax
constexpr int kQsStride = kHeadDim + 16;

struct MmaSmem {
  alignas(128) uint8_t slot[kMmaSlots][kSlotBytes];
  uint64_t full[kMmaSlots];
  uint64_t empty[kMmaSlots];
  uint64_t pairbar[kCons / 2];
  int rel[kMmaSlots];    // releases of the slot's current item (the second one refills it)
  int fills[kMmaSlots];  // copies issued into the slot
  int valid[kMmaSlots];
  int pt[kPtCache];
  alignas(16) uint32_t q[kGroup][kHeadDim / 2];  // the unit's query rows, bf16 pairs
  alignas(16) float qs[kGroup][kQsStride];       // the same rows as float, times a power of two
  float ep_m[kCons][kGroup];
  float ep_l[kCons][kGroup];
  int is_last;
  int abort;
};
static_assert(sizeof(MmaSmem) <= 227 * 1024, "shared memory per block");

// ----------------------------------------------------------------- PTX
__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// D (s32) += A (unsigned bytes, 16 x 32, row-major) * B (signed bytes, 32 x 8)
__device__ __forceinline__ void mma_u8s8(int (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.s32.u8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+r"(d[0]), "+r"(d[1]), "+r"(d[2]), "+r"(d[3])
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

// (lo, hi) -> packed pair, lo in the low half
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ float f16_lo(uint32_t w) {
  return __half2float(__ushort_as_half((unsigned short)(w & 0xffffu)));
}
__device__ __forceinline__ float f16_hi(uint32_t w) { return __half2float(__ushort_as_half((unsigned short)(w >> 16))); }

// Four stored code bytes (code + 128) -> two f16 pairs holding 1152 + code,
// exactly: each byte becomes the low mantissa byte of f16 1024 (0x6400 | b =
// 1024 + b).  lo = bytes 0, 1; hi = bytes 2, 3.
constexpr float kCodeOffset = 1152.f;
__device__ __forceinline__ void codes_to_f16(uint32_t w, uint32_t& lo, uint32_t& hi) {
  lo = __byte_perm(w, 0x64646464u, 0x5140);
  hi = __byte_perm(w, 0x64646464u, 0x5342);
}

// ----------------------------------------------------------------- copies in
// BF16 half-pages arrive by TMA as 128-byte-swizzled tiles: K at tiles 0-3 and V
// at tiles 4-7 of the slot (1024-byte aligned), tile c = channels 64c .. 64c+63
// of the 32 tokens, row r at byte 128 r, 16-byte chunk k stored at chunk k ^ (r % 8).
__device__ __forceinline__ uint8_t* bf16_tiles(uint8_t* slot) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(slot) + 1023) & ~uintptr_t(1023));
}
__device__ __forceinline__ uint32_t swz(int r, int chunk) {  // byte offset of (row, 16-byte chunk 0..31)
  return (chunk >> 3) * 4096 + r * 128 + (((chunk & 7) ^ (r & 7)) << 4);
}

// The page-table entry of item j: from the shared-memory copy, or from the global
// table for entries past the copy.
__device__ __forceinline__ int64_t item_slot(const DecodeParams& p, const UnitInfo& ui, const Items& it,
                                             const MmaSmem& S, int j) {
  const int page = item_page(ui, it, j);
  const int idx = page - it.pg_first;
  return idx < kPtCache ? S.pt[idx] : __ldg((ui.tier == 0 ? p.page_table : p.page_table8) + ui.pt_off + page);
}
// The page-table entry of item j straight from the global table (the first items
// are issued before the shared-memory copy exists).
__device__ __forceinline__ int64_t item_slot_global(const DecodeParams& p, const UnitInfo& ui, const Items& it, int j) {
  return __ldg((ui.tier == 0 ? p.page_table : p.page_table8) + ui.pt_off + item_page(ui, it, j));
}

// Issue the copy of item j, whose page-table entry is `slot`, into slot s.
__device__ __forceinline__ void mma_issue(const DecodeParams& p, const UnitInfo& ui, const Items& it, MmaSmem& S,
                                          int j, int s, int64_t slot) {
  int64_t lim = ui.tier == 0 ? p.kv_slots : p.rec_slots;
  const bool ok = slot >= 0 && (lim == 0 || slot < lim);
  S.valid[s] = ok;
  // test hook (tpk_set_test_wait): the chosen block's first item is neither copied
  // nor arrived on, so every wait on it runs out
  if (j == 0 && (int)blockIdx.x == p.stall_unit) return;
  if (!ok) {
    atomicOr(p.status, kStatusBadSlot);
    mbar_arrive(&S.full[s]);
    return;
  }
  if (ui.tier == 0) {
    const int row0 = (int)((slot * p.H + ui.h) * kPageTokens + ((it.first + j) & 1) * 32);
    uint8_t* base = bf16_tiles(S.slot[s]);
    mbar_arrive_expect_tx(&S.full[s], 32768);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      tma_load_2d(base + c * 4096, &p.kmap, 64 * c, row0, &S.full[s]);
      tma_load_2d(base + 16384 + c * 4096, &p.vmap, 64 * c, row0, &S.full[s]);
    }
  } else {
    const uint8_t* src = p.rec_pool + (slot * p.H + ui.h) * (int64_t)kRecordBytes;
    mbar_arrive_expect_tx(&S.full[s], kRecordBytes);
    bulk_g2s(S.slot[s], src, kRecordBytes, &S.full[s]);
  }
}

// Online-softmax update for this thread's base-2 scores x[] of query row g (-inf
// where masked).  Rescales O (rows 2t, 2t + 1) when a row maximum moved, turns
// x[] into weights and returns the factor alpha the row sum must be scaled by.
template <int N, int M>
__device__ __forceinline__ float softmax_rescale(float (&x)[N], float& m_run, float (&O)[M][4]) {
  const int lane = threadIdx.x & 31, t = lane & 3;
  float mx = kNegInf;
#pragma unroll
  for (int i = 0; i < N; ++i) mx = fmaxf(mx, x[i]);
  mx = fmaxf(mx, __shfl_xor_sync(kAll, mx, 1));
  mx = fmaxf(mx, __shfl_xor_sync(kAll, mx, 2));
  const float m_new = (mx == kNegInf) ? m_run : fmaxf(m_run, ceilf(mx));
  const float alpha = (m_new == m_run) ? 1.f : (m_run == kNegInf ? 0.f : ldexpf(1.f, (int)(m_run - m_new)));
  if (!__all_sync(kAll, alpha == 1.f)) {
    const float a0 = __shfl_sync(kAll, alpha, 8 * t);      // row 2t is held by lanes 4 * (2t) ..
    const float a1 = __shfl_sync(kAll, alpha, 8 * t + 4);  // row 2t + 1
#pragma unroll
    for (int m = 0; m < M; ++m) {
      O[m][0] *= a0;
      O[m][1] *= a1;
      O[m][2] *= a0;
      O[m][3] *= a1;
    }
  }
#pragma unroll
  for (int i = 0; i < N; ++i) x[i] = (x[i] == kNegInf) ? 0.f : exp2f(x[i] - m_new);
  m_run = m_new;
  return alpha;
}

// The two warps of a pair add up N partial scores per thread through shared
// memory: each writes its own values into `mine` (bytes of the slot that only it
// reads, and has finished reading), the pair meets at its mbarrier (a bounded
// wait: false if the partner did not arrive), and each adds the partner's values
// for the same lane (a + b = b + a, so both warps get the same sums).  Float4 k of
// lane l sits at row (32k + l) / 8, byte 16 (l % 8) of rows RowStride bytes apart.
struct PairSync {
  uint64_t* bar;    // the pair's mbarrier (count 2: one arrival per warp)
  uint32_t parity;  // phase of this item
  int* status;
  uint64_t limit;   // wait limit (ns)
};
template <int N, int RowStride>
__device__ __forceinline__ bool pair_exchange(float (&v)[N], uint8_t* mine, const uint8_t* theirs, const PairSync& ps) {
  const int lane = threadIdx.x & 31;
  __syncwarp();
#pragma unroll
  for (int k = 0; k < N / 4; ++k)
    *reinterpret_cast<float4*>(mine + ((32 * k + lane) >> 3) * RowStride + (lane & 7) * 16) =
        make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
  __syncwarp();
  if (lane == 0) mbar_arrive(ps.bar);
  if (!mbar_wait(ps.bar, ps.parity, ps.status, ps.limit)) return false;
#pragma unroll
  for (int k = 0; k < N / 4; ++k) {
    const float4 o = *reinterpret_cast<const float4*>(theirs + ((32 * k + lane) >> 3) * RowStride + (lane & 7) * 16);
    v[4 * k] += o.x;
    v[4 * k + 1] += o.y;
    v[4 * k + 2] += o.z;
    v[4 * k + 3] += o.w;
  }
  return true;
}

// Generic-proxy writes into a slot (the score exchange, zeroed rows) must be
// ordered before the next bulk copy refills the slot.
__device__ __forceinline__ void fence_slot_writes() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// ------------------------------------------------------- 8-bit record
// Warp half h of a pair owns channels 128h .. 128h + 127 of a whole record (64
// tokens).  QK leaves in x[k] the full (both halves) dot product of query row g
// with the codes of token 16t + k, before the per-token factor; the warp's partial
// scores over its channels are summed with the partner's through shared memory, so
// both warps hold the full scores and run the same softmax.  PV k-step i (0..3)
// covers tokens 16t + 4i + {0..3} of every thread t; the warp accumulates its 128
// channels.

// Float query: tile j (0..7) column 2t + e is token 16t + 2j + e; k-step 4J + i
// uses channels 128h + 64J + 16t + 4i + {0, 1} (k = 2t, 2t+1) and + {2, 3} (k =
// 2t+8, 2t+9).
__device__ __forceinline__ bool qk_float_query(uint8_t* rec, int h, const PairSync& psync, const MmaSmem& S,
                                               float (&x)[16]) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const float* ks = reinterpret_cast<const float*>(rec + kOffKsChan);
  const uint8_t* kc = rec + kOffKc;
  const float* qrow = S.qs[g];
  float acc[8][4];
#pragma unroll
  for (int j = 0; j < 8; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
  float qsum = 0.f;  // sum of this thread's 32 folded-query values of row g
#pragma unroll
  for (int J = 0; J < 2; ++J) {
    const int cb = 128 * h + 64 * J + 16 * t;
    uint4 kw[8];
#pragma unroll
    for (int j = 0; j < 8; ++j)  // token 16 (g >> 1) + 2j + (g & 1) (odd tokens: 64-byte halves swapped)
      kw[j] = *reinterpret_cast<const uint4*>(kc + (16 * (g >> 1) + 2 * j + (g & 1)) * kHeadDim + (cb ^ ((g & 1) << 6)));
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int ch = cb + 4 * i;
      const float4 s4 = *reinterpret_cast<const float4*>(ks + ks_index(ch));
      const float4 q4 = *reinterpret_cast<const float4*>(qrow + ks_index(ch));
      const float x0 = q4.x * s4.x, x1 = q4.y * s4.y, x2 = q4.z * s4.z, x3 = q4.w * s4.w;
      qsum += (x0 + x1) + (x2 + x3);
      const uint32_t h01 = pack_f16(x0, x1), h23 = pack_f16(x2, x3);
      const uint32_t l01 = pack_f16(x0 - f16_lo(h01), x1 - f16_hi(h01));
      const uint32_t l23 = pack_f16(x2 - f16_lo(h23), x3 - f16_hi(h23));
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint32_t w = i == 0 ? kw[j].x : i == 1 ? kw[j].y : i == 2 ? kw[j].z : kw[j].w;
        uint32_t b0, b1;
        codes_to_f16(w, b0, b1);
        mma_f16(acc[j], h01, l01, h23, l23, b0, b1);
      }
    }
  }
  // The products ran on 1152 + code: remove 1152 * sum_c q'_c over this warp's
  // channels (row g) from the high plane's dot before the low plane's is added.
  qsum += __shfl_xor_sync(kAll, qsum, 1);
  qsum += __shfl_xor_sync(kAll, qsum, 2);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    x[2 * j] = fmaf(-kCodeOffset, qsum, acc[j][0]) + acc[j][2];
    x[2 * j + 1] = fmaf(-kCodeOffset, qsum, acc[j][1]) + acc[j][3];
  }
  // partial scores of the two channel halves -> full scores in both warps (the
  // exchange area: rows 0..15 of this warp's half of the key codes)
  return pair_exchange<16, kHeadDim>(x, rec + kOffKc + 128 * h, rec + kOffKc + 128 * (h ^ 1), psync);
}

// Integer query ("SYCL", "Attention that reads 8-bit history": the integer query
// cache; the two-by-two experiment on which products run on integers).  Row g of
// q' = q s_c is coded per record with the absmax rule of the key codes: alpha =
// max_c |q'_c| / 127 over all 256 channels, codes rint(q'_c * (127 / max)), the
// divisions correctly rounded.  QK then runs on the integer tensor path with the
// operands swapped, so every row of the tile carries work: A = 16 tokens of stored
// key bytes (code + 128, unsigned), B = the 8 rows' query codes (signed), D = 16
// tokens x 8 rows in exact s32.  m-tile mt, row r is token 16mt + r; k-step (J, i2)
// uses channels 128h + 64J + 16t + 8i2 + {0..3} (k = 4t..4t+3) and + {4..7} (k =
// 16+4t..), the same 16 channels per thread as the float query.  The offset 128 is
// removed as 128 * sum_c qi_c; the partial dots of the two halves are added (exactly)
// through shared memory, transposed on the way to the score layout of the softmax.
constexpr float kRoundMagic = 12582912.f;  // 1.5 * 2^23
constexpr int kRoundMagicBits = 0x4B400000;  // its float32 encoding
__device__ __forceinline__ bool qk_int_query(uint8_t* rec, int h, const PairSync& psync, const MmaSmem& S,
                                             float (&x)[16]) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const float* ks = reinterpret_cast<const float*>(rec + kOffKsChan);
  const uint8_t* kc = rec + kOffKc;
  const float* qrow = S.qs[g];
  // q' of this thread's own channels, and the absmax over the whole row (the
  // partner half read contiguously: channels 128 (h ^ 1) + 16i + 4t)
  float y[2][4][4];
  float mx = 0.f;
#pragma unroll
  for (int J = 0; J < 2; ++J)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int ch = 128 * h + 64 * J + 16 * t + 4 * i;
      const float4 s4 = *reinterpret_cast<const float4*>(ks + ks_index(ch));
      const float4 q4 = *reinterpret_cast<const float4*>(qrow + ks_index(ch));
      y[J][i][0] = q4.x * s4.x;
      y[J][i][1] = q4.y * s4.y;
      y[J][i][2] = q4.z * s4.z;
      y[J][i][3] = q4.w * s4.w;
      mx = fmaxf(mx, fmaxf(fmaxf(fabsf(y[J][i][0]), fabsf(y[J][i][1])), fmaxf(fabsf(y[J][i][2]), fabsf(y[J][i][3]))));
    }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int ch = 128 * (h ^ 1) + 16 * i + 4 * t;
    const float4 s4 = *reinterpret_cast<const float4*>(ks + ks_index(ch));
    const float4 q4 = *reinterpret_cast<const float4*>(qrow + ks_index(ch));
    mx = fmaxf(mx, fmaxf(fmaxf(fabsf(q4.x * s4.x), fabsf(q4.y * s4.y)), fmaxf(fabsf(q4.z * s4.z), fabsf(q4.w * s4.w))));
  }
  mx = fmaxf(mx, __shfl_xor_sync(kAll, mx, 1));
  mx = fmaxf(mx, __shfl_xor_sync(kAll, mx, 2));
  const float inv = mx > 0.f ? __fdiv_rn(127.f, mx) : 0.f;
  const float alpha = __fdiv_rn(mx, 127.f);
  // codes, four to a word (channel order = byte order).  |y * inv| <= 127 (1 + 2^-24)
  // rounds to at most 127, so no clamp is needed.  Rounding to an integer by adding
  // 1.5 * 2^23 (the sum lands in [2^23, 2^24), where the float32 spacing is 1, so the
  // addition rounds half to even exactly like rint) leaves the code in the low bits
  // of the sum's encoding: its low byte is the code's two's-complement byte.
  uint32_t qw[2][4];
  int qsum = 0;
#pragma unroll
  for (int J = 0; J < 2; ++J)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t c[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) c[e] = __float_as_uint(__fadd_rn(__fmul_rn(y[J][i][e], inv), kRoundMagic));
      qw[J][i] = __byte_perm(__byte_perm(c[0], c[1], 0x0040), __byte_perm(c[2], c[3], 0x0040), 0x5410);
      qsum = __dp4a((int)qw[J][i], 0x01010101, qsum);
    }
  int acc[4][4];
#pragma unroll
  for (int mt = 0; mt < 4; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0;
#pragma unroll
  for (int J = 0; J < 2; ++J) {
    const int cb = (128 * h + 64 * J + 16 * t) ^ ((g & 1) << 6);  // tokens g, g + 8 share g's parity
#pragma unroll
    for (int mt = 0; mt < 4; ++mt) {
      const uint4 ka = *reinterpret_cast<const uint4*>(kc + (16 * mt + g) * kHeadDim + cb);
      const uint4 kb = *reinterpret_cast<const uint4*>(kc + (16 * mt + g + 8) * kHeadDim + cb);
      mma_u8s8(acc[mt], ka.x, kb.x, ka.y, kb.y, qw[J][0], qw[J][1]);
      mma_u8s8(acc[mt], ka.z, kb.z, ka.w, kb.w, qw[J][2], qw[J][3]);
    }
  }
  // sum_c qi_c of rows 2t and 2t + 1 over this warp's channels (the code offset)
  qsum += __shfl_xor_sync(kAll, qsum, 1);
  qsum += __shfl_xor_sync(kAll, qsum, 2);
  const int cq0 = 128 * __shfl_sync(kAll, qsum, 8 * t), cq1 = 128 * __shfl_sync(kAll, qsum, 8 * t + 4);
  // Exchange area: bytes 128h .. 128h + 127 of key-code rows 0..15 (codes only
  // this warp reads, and has read).  Dot (token tau, row rho) sits in row tau / 4,
  // word rho + 8 ((tau + tau / 16) mod 4): conflict-free both for the stores
  // (tau = 16mt + g (+ 8), rho = 2t, 2t + 1) and for the transposed loads (tau =
  // 16t + k, rho = g).
  uint8_t* mine = rec + kOffKc + 128 * h;
  const uint8_t* theirs = rec + kOffKc + 128 * (h ^ 1);
  __syncwarp();
#pragma unroll
  for (int mt = 0; mt < 4; ++mt)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int tau = 16 * mt + 8 * e + g;
      *reinterpret_cast<int2*>(mine + (tau >> 2) * kHeadDim + 4 * (2 * t + 8 * ((tau + mt) & 3))) =
          make_int2(acc[mt][2 * e] - cq0, acc[mt][2 * e + 1] - cq1);
    }
  __syncwarp();
  if (lane == 0) mbar_arrive(psync.bar);
  if (!mbar_wait(psync.bar, psync.parity, psync.status, psync.limit)) return false;
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    const int off = ((16 * t + k) >> 2) * kHeadDim + 4 * (g + 8 * ((k + t) & 3));
    const int d = *reinterpret_cast<const int*>(mine + off) + *reinterpret_cast<const int*>(theirs + off);
    // |d| <= 256 * 127 * 127 < 2^22: the encoding of 1.5 * 2^23 + d, minus 1.5 * 2^23,
    // is d as a float, exactly
    x[k] = __fmul_rn(__fsub_rn(__int_as_float(d + kRoundMagicBits), kRoundMagic), alpha);
  }
  return true;
}

template <bool IntQuery>
__device__ __forceinline__ bool process_int8_record(uint8_t* rec, int h, const PairSync& psync, const MmaSmem& S,
                                                    float qk_scale, float& m_run, float& l_run, float (&O)[8][4]) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const float* kr = reinterpret_cast<const float*>(rec + kOffKsTok);
  const float* vs = reinterpret_cast<const float*>(rec + kOffVsChan) + 128 * h;
  const uint8_t* vc = rec + kOffVc;
  float x[16];  // x[k]: token 16t + k
  if (IntQuery) {
    if (!qk_int_query(rec, h, psync, S, x)) return false;
  } else {
    if (!qk_float_query(rec, h, psync, S, x)) return false;
  }
  {
    // r_t of tokens 16t .. 16t + 15, then base-2 scores
    float rr[16];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float4 r4 = *reinterpret_cast<const float4*>(kr + 16 * t + 4 * k);
      rr[4 * k] = r4.x;
      rr[4 * k + 1] = r4.y;
      rr[4 * k + 2] = r4.z;
      rr[4 * k + 3] = r4.w;
    }
#pragma unroll
    for (int k = 0; k < 16; ++k) x[k] = x[k] * qk_scale * rr[k];
  }
  const float alpha = softmax_rescale<16, 8>(x, m_run, O);
  // P^T as one f16 plane: pw[k] = tokens 16t + 2k, 16t + 2k + 1 of row g.  The
  // rounded weights are the ones summed into l, so numerator and denominator
  // use the same probabilities.
  uint32_t pw[8];
  float lp = 0.f;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    pw[k] = pack_f16(x[2 * k], x[2 * k + 1]);
    lp += f16_lo(pw[k]) + f16_hi(pw[k]);
  }
  l_run = l_run * alpha + lp;
  // sum of the record's 64 weights of each row; the PV accumulator of rows 2t and
  // 2t + 1 starts at -1152 times it, cancelling the code offset
  float ps = lp + __shfl_xor_sync(kAll, lp, 1);
  ps += __shfl_xor_sync(kAll, ps, 2);
  const float c0 = -kCodeOffset * __shfl_sync(kAll, ps, 8 * t);
  const float c1 = -kCodeOffset * __shfl_sync(kAll, ps, 8 * t + 4);
  // ---- PV: this warp's 8 channel tiles, 4 k-steps of 16 tokens; each page's
  // result times u_c into the accumulator
#pragma unroll
  for (int m = 0; m < 8; ++m) {
    const int ch = 128 * h + 16 * m + g;
    const uint4 va = *reinterpret_cast<const uint4*>(vc + vc_byte(ch, 16 * t));
    const uint4 vb = *reinterpret_cast<const uint4*>(vc + vc_byte(ch + 8, 16 * t));
    float c[4] = {c0, c1, c0, c1};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t a0, a2, a1, a3;
      codes_to_f16(i == 0 ? va.x : i == 1 ? va.y : i == 2 ? va.z : va.w, a0, a2);
      codes_to_f16(i == 0 ? vb.x : i == 1 ? vb.y : i == 2 ? vb.z : vb.w, a1, a3);
      mma_f16(c, a0, a1, a2, a3, pw[2 * i], pw[2 * i + 1]);
    }
    const float ua = vs[16 * m + g], ub = vs[16 * m + g + 8];
    O[m][0] = fmaf(ua, c[0], O[m][0]);
    O[m][1] = fmaf(ua, c[1], O[m][1]);
    O[m][2] = fmaf(ub, c[2], O[m][2]);
    O[m][3] = fmaf(ub, c[3], O[m][3]);
  }
  return true;
}

// ------------------------------------------------------ BF16 half page
// Warp half h of a pair owns channels 128h .. 128h + 127 of a BF16 half-page item
// (32 tokens, K at tiles 0-3 and V at tiles 4-7 of the slot).  QK tile j (0..3)
// column 2t + e is token 8j + 2t + e of the item; the partial scores over the
// warp's channels are exchanged as for the 8-bit tier.  PV k-step i (0..1)
// covers tokens 16i .. 16i + 15.
__device__ __forceinline__ bool process_bf16_half(uint8_t* slot, int h, const PairSync& psync, int tok0, int tb,
                                                  int te, const MmaSmem& S, float qscale, float& m_run, float& l_run,
                                                  float (&O)[8][4]) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  uint8_t* K = bf16_tiles(slot);
  uint8_t* V = K + 16384;
  if (tok0 < tb || tok0 + 32 > te) {  // zero this warp's value channels of tokens outside the range
    for (int r0 = 0; r0 < 32; r0 += 2) {
      const int r = r0 + (lane >> 4), tok = tok0 + r;
      if (tok < tb || tok >= te)
        *reinterpret_cast<uint4*>(V + (2 * h + ((lane >> 3) & 1)) * 4096 + r * 128 + (lane & 7) * 16) =
            make_uint4(0, 0, 0, 0);
    }
    __syncwarp();
  }
  const uint32_t* qrow = S.q[g];
  float acc[4][4];
#pragma unroll
  for (int j = 0; j < 4; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
#pragma unroll
  for (int kq = 0; kq < 4; ++kq) {
    const int kk = 4 * h + kq;  // 32 channels 32kk .. 32kk + 31
    const uint32_t qa0 = qrow[16 * kk + t], qa1 = qrow[16 * kk + 4 + t];
    const uint32_t qa2 = qrow[16 * kk + 8 + t], qa3 = qrow[16 * kk + 12 + t];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t m4[4];
      ldsm_x4(m4, K + swz(8 * j + (lane & 7), 4 * kk + (lane >> 3)));
      mma_bf16(acc[j], qa0, 0u, qa1, 0u, m4[0], m4[1]);
      mma_bf16(acc[j], qa2, 0u, qa3, 0u, m4[2], m4[3]);
    }
  }
  float x[8];  // x[2j + e]: token 8j + 2t + e of the item
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    x[2 * j] = acc[j][0];
    x[2 * j + 1] = acc[j][1];
  }
  // exchange area: the first 1 KB of this warp's key tiles (2h, 2h + 1)
  if (!pair_exchange<8, 128>(x, K + 2 * h * 4096, K + 2 * (h ^ 1) * 4096, psync)) return false;
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int tok = tok0 + 8 * j + 2 * t + e;
      x[2 * j + e] = (tok >= tb && tok < te) ? x[2 * j + e] * qscale : kNegInf;
    }
  {
    const float alpha = softmax_rescale<8, 8>(x, m_run, O);
    l_run = l_run * alpha + (((x[0] + x[1]) + (x[2] + x[3])) + ((x[4] + x[5]) + (x[6] + x[7])));
  }
  // P^T for k-step i: tokens 16i + 2t + {0, 1} (tile 2i) and 16i + 8 + 2t + {0, 1}
  // (tile 2i + 1), as bf16 high and low planes
  const int mi = lane >> 3;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const uint32_t ph0 = pack_bf16(x[4 * i], x[4 * i + 1]), ph1 = pack_bf16(x[4 * i + 2], x[4 * i + 3]);
    const uint32_t pl0 = pack_bf16(x[4 * i] - bf16_lo(ph0), x[4 * i + 1] - bf16_hi(ph0));
    const uint32_t pl1 = pack_bf16(x[4 * i + 2] - bf16_lo(ph1), x[4 * i + 3] - bf16_hi(ph1));
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      uint32_t a[4];
      ldsm_x4_t(a, V + swz(16 * i + (mi >> 1) * 8 + (lane & 7), 2 * (8 * h + m) + (mi & 1)));
      mma_bf16(O[m], a[0], a[1], a[2], a[3], ph0, ph1);
      mma_bf16(O[m], a[0], a[1], a[2], a[3], pl0, pl1);
    }
  }
  return true;
}

// ------------------------------------------------------------------ kernel
template <int R, bool IntQuery>
__global__ void __launch_bounds__(kMmaThreads, 1) decode_mma_kernel(const __grid_constant__ DecodeParams p,
                                                                  const __grid_constant__ Plan<R> plan) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  MmaSmem& S = *reinterpret_cast<MmaSmem*>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t = lane & 3;

  const UnitInfo ui = decode_unit(p, plan.req, blockIdx.x);
  const Items it = unit_items(ui);
  // One thread (the block's last) sets up the barriers and issues the copies; the
  // others meanwhile bring the unit's page-table entries and query rows into
  // shared memory, so the two memory round trips of the start overlap.
  constexpr int kIssuer = kMmaThreads - 1;
  if (tid == kIssuer) {
    for (int s = 0; s < kMmaSlots; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], 2);
    }
    for (int q = 0; q < kCons / 2; ++q) mbar_init(&S.pairbar[q], 2);
    for (int s = 0; s < kMmaSlots; ++s) S.rel[s] = S.fills[s] = 0;
    S.abort = 0;
    fence_mbar_init();
    // The first three items go out at once, straight from the global page table
    // (their entries loaded together first: one memory round trip); the next
    // three as soon as the page table is in shared memory, and every later item
    // is issued by the warp that releases its slot's previous item last.  (All six
    // at once made every block's first record land later: measured 0.9 µs slower
    // per 128K step.)
    int64_t first[kFirstIssue];
#pragma unroll
    for (int j = 0; j < kFirstIssue; ++j) first[j] = j < it.n ? item_slot_global(p, ui, it, j) : 0;
#pragma unroll
    for (int j = 0; j < kFirstIssue; ++j)
      if (j < it.n) {
        mma_issue(p, ui, it, S, j, j, first[j]);
        S.fills[j] = 1;
      }
  } else {
    const int32_t* pt = (ui.tier == 0 ? p.page_table : p.page_table8) + ui.pt_off + it.pg_first;
    const int n = min(it.n_pages, kPtCache);
    for (int i = tid; i < n; i += kMmaThreads - 1) S.pt[i] = __ldg(pt + i);
    const uint4* q128 = reinterpret_cast<const uint4*>(p.q + (int64_t)(ui.b * p.H + ui.h) * kGroup * kHeadDim);
    for (int i = tid; i < kGroup * kHeadDim / 8; i += kMmaThreads - 1)
      reinterpret_cast<uint4*>(&S.q[0][0])[i] = __ldg(q128 + i);
  }
  __syncthreads();
  // 8-bit tier: a float copy of q times 2^-(e+1), e the exponent of the row's max
  // |q|: with s_c <= 2^14 every q'_c = q_c s_c of this row then stays below 2^13,
  // inside f16 range, whatever the page.  Thread (g, t) of every warp reads a
  // quarter of row g with 16-byte loads for the row maximum; warp w writes
  // channels 32w .. 32w + 31 of the float copy.  (The exact tier reads the bf16
  // rows as they are and starts at once.)
  float qk_scale = p.qscale;
  if (ui.tier == 1) {
    float qmax = 0.f;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint4 w = *reinterpret_cast<const uint4*>(&S.q[g][4 * (t + 4 * k)]);
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) qmax = fmaxf(qmax, fmaxf(fabsf(bf16_lo(ws[e])), fabsf(bf16_hi(ws[e]))));
    }
    qmax = fmaxf(qmax, __shfl_xor_sync(kAll, qmax, 1));
    qmax = fmaxf(qmax, __shfl_xor_sync(kAll, qmax, 2));
    int e = 0;
    frexpf(qmax, &e);
    const float sc = qmax > 0.f ? ldexpf(1.f, -(e + 1)) : 1.f;
    qk_scale = p.qscale / sc;
    // lane (g, t): row g, channels 32 warp + 8 t .. + 7 (every lane of row g holds
    // the row's scale)
    const uint4 w = *reinterpret_cast<const uint4*>(&S.q[g][16 * warp + 4 * t]);
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int e2 = 0; e2 < 4; ++e2) {
      const int c = 32 * warp + 8 * t + 2 * e2;
      S.qs[g][ks_index(c)] = bf16_lo(ws[e2]) * sc;  // same channel permutation as the record's s_c
      S.qs[g][ks_index(c + 1)] = bf16_hi(ws[e2]) * sc;
    }
    __syncthreads();
  }
  // The next three items.  (Issuing a copy can stall its thread while earlier
  // copies are still under way, so this comes after the block-wide steps: only
  // the issuer's own warp waits, and its pair's first item is among these.)
  if (tid == kIssuer) {
    for (int j = kFirstIssue; j < min(it.n, kMmaSlots); ++j) {
      mma_issue(p, ui, it, S, j, j, item_slot(p, ui, it, S, j));
      S.fills[j] = 1;
    }
  }

  float O[8][4];  // this warp's 128 channels of the pair's output
#pragma unroll
  for (int m = 0; m < 8; ++m) O[m][0] = O[m][1] = O[m][2] = O[m][3] = 0.f;
  float m_run = kNegInf, l_run = 0.f;

  {
    const int pair = warp >> 1, half = warp & 1;
    uint32_t pair_phase = 0;  // items this pair has exchanged scores for (both warps skip the same items)
    for (int j = pair; j < it.n; j += kCons / 2) {
      const int s = j % kMmaSlots;
      // Slot s last held item j - 6, which another pair may still own.  A parity
      // wait on full[s] would then match that item's phase, so first wait for its
      // release (empty[s] is at most one phase behind here: item j - 12 belonged
      // to this pair), after which full[s]'s pending phase is item j's.
      if (j >= kMmaSlots && !mbar_wait(&S.empty[s], ((j / kMmaSlots) - 1) & 1, p.status, p.wait_ns)) {
        S.abort = 1;
        break;
      }
      if (!mbar_wait(&S.full[s], (j / kMmaSlots) & 1, p.status, p.wait_ns)) {
        S.abort = 1;
        break;
      }
      if (S.valid[s]) {
        const PairSync psync{&S.pairbar[pair], pair_phase & 1, p.status, p.wait_ns};
        ++pair_phase;
        const bool ok = ui.tier == 1
                            ? process_int8_record<IntQuery>(S.slot[s], half, psync, S, qk_scale, m_run, l_run, O)
                            : process_bf16_half(S.slot[s], half, psync, (it.first + j) * 32, ui.tok_begin,
                                                ui.tok_end, S, p.qscale, m_run, l_run, O);
        if (!ok) {
          S.abort = 1;
          break;
        }
        fence_slot_writes();
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&S.empty[s]);
        // the second warp of the pair to let go of the slot refills it
        if (j + kMmaSlots < it.n) {
          __threadfence_block();
          if (atomicAdd(&S.rel[s], 1) == 1) {
            S.rel[s] = 0;
            __threadfence_block();
            mma_issue(p, ui, it, S, j + kMmaSlots, s, item_slot(p, ui, it, S, j + kMmaSlots));
            S.fills[s] += 1;
          }
        }
      }
    }
  }
  __syncthreads();
  if (S.abort) {
    // A wait gave up: let every copy issued into the slots land (bounded: the
    // latest fill of each slot), then leave without a result; the status word
    // reports the timeout.
    if (tid == 0)
      for (int s = 0; s < kMmaSlots; ++s)
        if (S.fills[s] > 0) mbar_wait(&S.full[s], (S.fills[s] - 1) & 1, p.status, p.wait_ns);
    __syncthreads();
    return;
  }
  // ---- per-pair states into shared memory (the stages are idle now); the two
  // warps of a pair hold the same softmax state and one channel half each
  // [4 pairs][8 rows][kEpStride]: rows padded by 4 floats so that the scattered
  // accumulator stores (rows 2t, 2t + 1 of lane (g, t)) hit distinct banks
  constexpr int kEpStride = kHeadDim + 4;
  float* ep_o = reinterpret_cast<float*>(S.slot[0]);
  if (warp < kCons) {
    const int pair = warp >> 1, half = warp & 1;
    float L = l_run;
    L += __shfl_xor_sync(kAll, L, 1);
    L += __shfl_xor_sync(kAll, L, 2);
    if (t == 0 && half == 0) {
      S.ep_m[pair][g] = m_run;
      S.ep_l[pair][g] = L;
    }
    float* base = ep_o + pair * kGroup * kEpStride + 128 * half;
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      base[(2 * t) * kEpStride + 16 * m + g] = O[m][0];
      base[(2 * t + 1) * kEpStride + 16 * m + g] = O[m][1];
      base[(2 * t) * kEpStride + 16 * m + g + 8] = O[m][2];
      base[(2 * t + 1) * kEpStride + 16 * m + g + 8] = O[m][3];
    }
  }
  __syncthreads();
  write_and_fold<kCons / 2, MmaSmem, kEpStride>(p, ui, S, ep_o);
}

template <int R, bool IntQuery>
static cudaError_t launch_mma(const DecodeParams& p, const ReqPlan* req, cudaStream_t stream) {
  static DeviceOnce once;
  const int smem = (int)sizeof(MmaSmem);
  cudaError_t e = once.run([&] {
    return cudaFuncSetAttribute(decode_mma_kernel<R, IntQuery>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  });
  if (e != cudaSuccess) return e;
  Plan<R> plan = {};
  for (int b = 0; b < p.n_req; ++b) plan.req[b] = req[b];
  decode_mma_kernel<R, IntQuery><<<p.n_units, kMmaThreads, smem, stream>>>(p, plan);
  return cudaGetLastError();
}

cudaError_t launch_decode_mma(const DecodeParams& p, const ReqPlan* req, cudaStream_t stream) {
  if (p.n_units == 0) return cudaSuccess;
  if (p.int_query)
    return p.n_req <= kShortPlan ? launch_mma<kShortPlan, true>(p, req, stream)
                                 : launch_mma<kMaxReqPerLaunch, true>(p, req, stream);
  return p.n_req <= kShortPlan ? launch_mma<kShortPlan, false>(p, req, stream)
                               : launch_mma<kMaxReqPerLaunch, false>(p, req, stream);
}

int decode_mma_blocks_per_sm() {
  int n = 0;
  const int smem = (int)sizeof(MmaSmem);
  cudaFuncSetAttribute(decode_mma_kernel<kMaxReqPerLaunch, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_mma_kernel<kMaxReqPerLaunch, false>, kMmaThreads,
                                                    smem) !=
      cudaSuccess)
    return 1;
  return n > 0 ? n : 1;
}

}  // namespace tpk
