// Device-side helpers shared by the tpk kernels: sizes of the page formats,
// mbarrier and bulk-copy (cp.async.bulk) wrappers written as inline PTX for
// sm_103a, and the per-launch split plan passed by value to the decode kernels.
#pragma once
#include <cuda.h>  // CUtensorMap (type only; the encode entry point is fetched at run time)
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <mutex>

namespace tpk {

constexpr int kHeadDim = 256;
constexpr int kPageTokens = 64;
constexpr int kGroup = 8;  // query rows per KV head
constexpr int kRecordBytes = 35072;
constexpr int kOffKc = 0;
constexpr int kOffVc = 16384;
constexpr int kOffKsChan = 32768;
constexpr int kOffKsTok = 33792;
constexpr int kOffVsChan = 34048;
constexpr int kBf16PageHeadBytes = kPageTokens * kHeadDim * 2;  // 32 KB (K or V)

// Position swizzles of the record fields (they spread the tensor-core kernel's
// shared-memory reads over all banks):
//   key code (t, c)   at byte t*256 + (c ^ 64 (t & 1))
//   value code (c, t) at byte c*64 + (t ^ 32 ((c >> 1) & 1))
//   s_c               at float c ^ 8 ((c >> 5) & 1)
__host__ __device__ __forceinline__ int kc_byte(int t, int c) { return t * kHeadDim + (c ^ ((t & 1) << 6)); }
__host__ __device__ __forceinline__ int vc_byte(int c, int t) { return c * kPageTokens + (t ^ (((c >> 1) & 1) << 5)); }
__host__ __device__ __forceinline__ int ks_index(int c) { return c ^ (((c >> 5) & 1) << 3); }

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Device status bits (read by tpk_get_device_status).
constexpr int kStatusBadSlot = 1;

// ----------------------------------------------------------------- split plan
// One request's share of a decode launch.  Thread block u belongs to the request
// with the largest unit_base <= u; within the request, units are laid out
// [kv_head][exact splits..., 8-bit splits...], so the units of one (request,
// head) are consecutive and are folded in that order.
struct ReqPlan {
  int32_t unit_base;  // first unit of this request
  int32_t pt_off;     // offset of the request's exact-tier slots in page_table
  int32_t e_begin;    // exact-tier token range [e_begin, e_end)
  int32_t e_end;
  int32_t pt_off8;    // offset of the request's 8-bit slots in page_table8
  int32_t p_begin;    // 8-bit page range [p_begin, p_end)
  int32_t p_end;
  int16_t splits_e;   // exact-tier units per KV head (0 if the tier is empty)
  int16_t splits_8;   // 8-bit units per KV head
};

constexpr int kMaxReqPerLaunch = 256;
// Launches of at most kShortPlan requests pass a short plan: the kernels take
// the plan as a parameter, and a smaller parameter block is set up faster at
// every launch.
constexpr int kShortPlan = 4;
template <int R>
struct Plan {
  ReqPlan req[R];
};

enum : int { kModePrimitive = 0, kModeFold = 1 };

struct DecodeParams {
  CUtensorMap kmap;         // BF16 pools as 2-D tensors [slot * H * 64][256], 32 x 64 boxes,
  CUtensorMap vmap;         // 128-byte swizzle (tensor-core kernel only)
  const uint16_t* q;        // bf16 [n_req][H*G][256]
  const uint16_t* k_pool;   // bf16 [slot][H][64][256]
  const uint16_t* v_pool;
  const uint8_t* rec_pool;  // records [slot][H]
  const int32_t* page_table;
  const int32_t* page_table8;
  int64_t kv_slots;         // 0 = unchecked
  int64_t rec_slots;
  float* part_o;            // primitive: o_part [split][H*G][256]; multi-request: workspace [unit][G][256]
  float* part_lse;
  float* out_o;             // multi-request: final o [n_req][H*G][256]
  float* out_lse;
  int* status;              // device status word
  float qscale;             // sm_scale * log2(e)
  int int_query;            // 1: the 8-bit tier's QK runs on the integer query
  int H;
  int mode;
  int n_req;
  int n_units;
  uint64_t wait_ns;         // limit of every bounded wait (kWaitLimitNs unless a test sets it)
  int stall_unit;           // test hook: this block's first item is never issued (-1: none)
};

struct UnitInfo {
  int b, h, tier, split, n_splits, per_head, unit_in_head;
  int tok_begin, tok_end;  // exact tier: tokens; 8-bit tier: tokens of whole pages (page * 64)
  int pt_off;
};

__device__ __forceinline__ UnitInfo decode_unit(const DecodeParams& p, const ReqPlan* req, int u) {
  int lo = 0, hi = p.n_req - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (req[mid].unit_base <= u) lo = mid; else hi = mid - 1;
  }
  const ReqPlan& r = req[lo];
  UnitInfo ui;
  ui.b = lo;
  int local = u - r.unit_base;
  ui.per_head = r.splits_e + r.splits_8;
  ui.h = local / ui.per_head;
  int k = local - ui.h * ui.per_head;
  ui.unit_in_head = k;
  if (k < r.splits_e) {
    ui.tier = 0;
    ui.split = k;
    ui.n_splits = r.splits_e;
    // the exact tier is cut on page boundaries for the primitive call (its
    // documented pieces) and on half-page boundaries (the kernels' item) in the
    // multi-request launch, where finer cuts even out the units' lengths
    const int gran = p.mode == kModePrimitive ? kPageTokens : kPageTokens / 2;
    int pg0 = r.e_begin / gran;
    int pg1 = (r.e_end + gran - 1) / gran;
    int P = pg1 - pg0;
    int pa = pg0 + (int)((int64_t)P * k / r.splits_e);
    int pb = pg0 + (int)((int64_t)P * (k + 1) / r.splits_e);
    ui.tok_begin = max(r.e_begin, pa * gran);
    ui.tok_end = min(r.e_end, pb * gran);
    if (ui.tok_end < ui.tok_begin) ui.tok_end = ui.tok_begin;
    ui.pt_off = r.pt_off;
  } else {
    ui.tier = 1;
    ui.split = k - r.splits_e;
    ui.n_splits = r.splits_8;
    int P = r.p_end - r.p_begin;
    int pa = r.p_begin + (int)((int64_t)P * ui.split / r.splits_8);
    int pb = r.p_begin + (int)((int64_t)P * (ui.split + 1) / r.splits_8);
    ui.tok_begin = pa * kPageTokens;
    ui.tok_end = pb * kPageTokens;
    ui.pt_off = r.pt_off8;
  }
  return ui;
}

// Page conversion launch parameters (given-scale arrays are null for a full
// conversion).
// 13-bit lossless records (pack13.cu)
constexpr int kStatusBadRecord = 4;

struct Pack13Params {
  const uint16_t* k_pool;
  const uint16_t* v_pool;
  const int32_t* src;
  const int32_t* dst;
  uint8_t* out;
  int64_t kv_slots;   // 0 = unchecked
  int64_t out_slots;  // 0 = unchecked
  int* status;
  int H;
};

struct Unpack13Params {
  const uint8_t* src;
  const int64_t* offsets;  // per page-head, bytes
  int64_t src_bytes;       // 0 = unchecked
  const int32_t* dst;
  uint16_t* k_pool;
  uint16_t* v_pool;
  int64_t kv_slots;  // 0 = unchecked
  int* status;
  int H;
};

cudaError_t launch_pack13(const Pack13Params& p, int n_pages, cudaStream_t stream);
cudaError_t launch_unpack13(const Unpack13Params& p, int n_pages, cudaStream_t stream);

struct QuantParams {
  const uint16_t* k_pool;
  const uint16_t* v_pool;
  const int32_t* src;
  const int32_t* dst;
  uint8_t* rec_pool;
  const float* g_kchan;  // given scales, or null
  const float* g_ktok;
  const float* g_vchan;
  int64_t kv_slots;
  int64_t rec_slots;
  int* status;
  int H;
};

// --------------------------------------------------- per-device host state
// Kernel attributes (the dynamic shared-memory limit) and constant tables belong
// to a device's context, so one-time setup runs once per device, not once per
// process; several host threads may launch at once.
constexpr int kMaxDevices = 64;

class DeviceOnce {
 public:
  // Runs setup() for the current device unless it has succeeded there before; a
  // failed setup is retried by the next call.
  template <class F>
  cudaError_t run(F&& setup) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (done_[dev].load(std::memory_order_acquire)) return cudaSuccess;
    std::lock_guard<std::mutex> lock(mu_);
    if (done_[dev].load(std::memory_order_relaxed)) return cudaSuccess;
    e = setup();
    if (e == cudaSuccess) done_[dev].store(true, std::memory_order_release);
    return e;
  }

 private:
  std::mutex mu_;
  std::atomic<bool> done_[kMaxDevices] = {};
};

// A positive int per device, computed on first use (0: not known yet).  Racing
// first calls compute the same value.
template <class F>
int per_device_int(std::atomic<int> (&cache)[kMaxDevices], F&& compute) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return compute();
  int v = cache[dev].load(std::memory_order_relaxed);
  if (v <= 0) {
    v = compute();
    cache[dev].store(v, std::memory_order_relaxed);
  }
  return v;
}

// ------------------------------------------------------------- PTX wrappers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait on an mbarrier phase: gives up after limit_ns of wall time (two
// seconds unless a launch passes its own limit), sets kStatusTimeout in the
// device status word and returns false.
constexpr int kStatusTimeout = 2;
constexpr uint64_t kWaitLimitNs = 2000000000ull;
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int* status,
                                          uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (;;) {
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 > limit_ns) {
      atomicOr(status, kStatusTimeout);
      return false;
    }
  }
}

// 2-D tensor copy global -> shared (TMA), completion counted on an mbarrier.
// x is the innermost coordinate (elements), y the row.
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(smem_dst)),
      "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// 1-D bulk copy global -> shared, completion counted on an mbarrier (bytes and
// both addresses must be multiples of 16).
__device__ __forceinline__ void bulk_g2s(void* smem_dst, const void* gmem_src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(smem_dst)),
      "l"(gmem_src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}


__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

}  // namespace tpk
