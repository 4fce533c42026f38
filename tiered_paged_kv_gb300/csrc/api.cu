// Host side of the tpk C ABI: argument validation, the split planner and the
// kernel launches.  Every entry point validates before launching and reports
// failures as a tpk_status plus a thread-local message.
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "common.cuh"
#include "tpk.h"

namespace tpk {
cudaError_t launch_decode_simt(const DecodeParams& p, const ReqPlan* req, cudaStream_t stream);
int decode_simt_blocks_per_sm();
cudaError_t launch_decode_mma(const DecodeParams& p, const ReqPlan* req, cudaStream_t stream);
int decode_mma_blocks_per_sm();
cudaError_t launch_merge(int n_parts, int rows, const float* o_parts, const float* lse_parts, float* o_acc,
                         float* lse_acc, cudaStream_t stream);
cudaError_t launch_quantize(const QuantParams& p, int n_pages, cudaStream_t stream);
cudaError_t launch_fold(const DecodeParams& p, const ReqPlan* req, cudaStream_t stream);
}  // namespace tpk

using namespace tpk;

__device__ int g_tpk_status;

namespace tpk {
void set_error(const char* msg);
}

namespace {

constexpr int kMaxUnits = 2048;       // partial slots in the hybrid workspace (256 requests x 4 heads x 2 tiers)
constexpr int kMaxSplits = 4096;      // primitive calls
constexpr int kMaxHeads = 1024;

thread_local std::string g_err;

tpk_status fail(tpk_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_err = buf;
  return s;
}

tpk_status cuda_fail(cudaError_t e, const char* what) {
  return fail(TPK_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

tpk_status check_shape(const tpk_shape* s) {
  if (!s) return fail(TPK_ERR_INVALID, "shape is null");
  if (s->kv_heads < 1 || s->kv_heads > kMaxHeads) return fail(TPK_ERR_INVALID, "kv_heads %d out of [1, %d]", s->kv_heads, kMaxHeads);
  if (s->group != kGroup) return fail(TPK_ERR_UNSUPPORTED, "group %d (only 8 supported)", s->group);
  if (s->head_dim != kHeadDim) return fail(TPK_ERR_UNSUPPORTED, "head_dim %d (only 256 supported)", s->head_dim);
  if (s->page_tokens != kPageTokens) return fail(TPK_ERR_UNSUPPORTED, "page_tokens %d (only 64 supported)", s->page_tokens);
  if (!(s->sm_scale == 0.f || s->sm_scale == 0.0625f))
    return fail(TPK_ERR_UNSUPPORTED, "sm_scale %g (only 1/sqrt(256) supported)", (double)s->sm_scale);
  if (s->impl < TPK_IMPL_DEFAULT || s->impl > TPK_IMPL_TENSOR) return fail(TPK_ERR_INVALID, "impl %d", s->impl);
  if (s->kv_slots < 0 || s->rec_slots < 0) return fail(TPK_ERR_INVALID, "negative pool size");
  if (s->int_query != 0 && s->int_query != 1) return fail(TPK_ERR_INVALID, "int_query %d (0 or 1)", s->int_query);
  if (s->int_query && s->impl == TPK_IMPL_SIMT)
    return fail(TPK_ERR_UNSUPPORTED, "the integer query runs on the tensor-core kernel only");
  return TPK_OK;
}

int* status_ptr() {
  static std::atomic<int*> ptrs[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  int* q = ptrs[dev].load(std::memory_order_relaxed);
  if (!q) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_tpk_status) != cudaSuccess) return nullptr;
    q = static_cast<int*>(p);
    ptrs[dev].store(q, std::memory_order_relaxed);
  }
  return q;
}

int num_sms() {
  static std::atomic<int> cached[kMaxDevices] = {};
  return per_device_int(cached, [] {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    return n > 0 ? n : 1;
  });
}

// Test hook of the bounded waits (tpk_set_test_wait).
std::atomic<uint64_t> g_test_wait_ns{0};
std::atomic<int> g_test_stall_unit{-1};

void fill_common(DecodeParams& p, const tpk_shape* s, const void* q) {
  std::memset(&p, 0, sizeof(p));
  const uint64_t w = g_test_wait_ns.load(std::memory_order_relaxed);
  p.wait_ns = w > 0 ? w : kWaitLimitNs;
  p.stall_unit = g_test_stall_unit.load(std::memory_order_relaxed);
  p.q = static_cast<const uint16_t*>(q);
  p.kv_slots = s->kv_slots;
  p.rec_slots = s->rec_slots;
  p.qscale = 0.0625f * kLog2e;
  p.int_query = s->int_query;
  p.H = s->kv_heads;
}

bool use_simt(const tpk_shape* s) { return s->impl == TPK_IMPL_SIMT; }

// cuTensorMapEncodeTiled, fetched from the driver at run time (no link-time
// dependency on libcuda).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static std::atomic<EncodeTiledFn> fn{nullptr};
  EncodeTiledFn f = fn.load(std::memory_order_relaxed);
  if (!f) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess) {
      f = reinterpret_cast<EncodeTiledFn>(ptr);
      fn.store(f, std::memory_order_relaxed);
    }
  }
  return f;
}

// The tensor-core kernel reads BF16 half-pages with TMA: each pool is a 2-D
// tensor of [kv_slots * H * 64 rows][256 bf16] with 32-row x 64-column boxes and
// the 128-byte swizzle.
tpk_status make_pool_maps(DecodeParams& p, const tpk_shape* s, const void* k_pool, const void* v_pool) {
  if (use_simt(s)) return TPK_OK;
  if (s->kv_slots <= 0)
    return fail(TPK_ERR_INVALID, "kv_slots must be set: the tensor-core kernel reads the BF16 pools with TMA");
  const uint64_t rows = (uint64_t)s->kv_slots * s->kv_heads * kPageTokens;
  if (rows >= (1ull << 31)) return fail(TPK_ERR_UNSUPPORTED, "BF16 pool too large for one tensor map");
  EncodeTiledFn fn = encode_fn();
  if (!fn) return fail(TPK_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t dims[2] = {(cuuint64_t)kHeadDim, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)kHeadDim * 2};
  cuuint32_t box[2] = {64, 32};
  cuuint32_t estr[2] = {1, 1};
  const void* pools[2] = {k_pool, v_pool};
  CUtensorMap* maps[2] = {&p.kmap, &p.vmap};
  for (int i = 0; i < 2; ++i) {
    CUresult r = fn(maps[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(pools[i]), dims, strides, box,
                    estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(TPK_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  }
  return TPK_OK;
}

int blocks_per_sm(const tpk_shape* s) {
  static std::atomic<int> simt[kMaxDevices] = {}, mma[kMaxDevices] = {};
  if (use_simt(s)) return per_device_int(simt, decode_simt_blocks_per_sm);
  return per_device_int(mma, decode_mma_blocks_per_sm);
}

// Split plan of the multi-request call: cnt[2b] / cnt[2b + 1] = units per KV head
// of request b's exact / 8-bit tier.  Every request's heads share one split of
// each tier.  The U = waves * per_wave / H unit budget per head (waves: the fewest
// whole waves of resident blocks giving every segment about 4 units) is shared
// among the (request, tier) segments in proportion to their bytes (largest
// remainder, at least one unit per non-empty segment, at most one per page), so
// units carry about equal bytes and whole waves of resident blocks are filled.
tpk_status plan_splits(int H, int n_req, const int32_t* n_exact_tokens, const int32_t* n_int8_pages, int per_wave,
                       std::vector<int>& cnt) {
  int min_units = 0;
  for (int b = 0; b < n_req; ++b) min_units += std::max(1, (n_exact_tokens[b] > 0) + (n_int8_pages[b] > 0));
  if (min_units * H > kMaxUnits)
    return fail(TPK_ERR_UNSUPPORTED, "%d (request, head, tier) segments exceed %d units", min_units * H, kMaxUnits);
  // enough waves that segments average at least 4 units (balance across requests)
  const int want = std::max((per_wave + H - 1) / H, 4 * min_units) * H;
  const int waves = std::max(1, (want + per_wave - 1) / per_wave);
  const int U = std::max(min_units, std::min(kMaxUnits, waves * per_wave) / H);
  std::vector<double> wgt(2 * n_req);
  std::vector<int> cap(2 * n_req);
  cnt.assign(2 * n_req, 0);
  double W = 0.0;
  for (int b = 0; b < n_req; ++b) {
    const int ne = n_exact_tokens[b], n8 = n_int8_pages[b];
    wgt[2 * b] = 1024.0 * ne;
    wgt[2 * b + 1] = (double)kRecordBytes * n8;
    cap[2 * b] = ne > 0 ? (ne + kPageTokens - 1) / kPageTokens : (n8 > 0 ? 0 : 1);  // empty request: one empty unit
    cap[2 * b + 1] = n8;
    W += wgt[2 * b] + wgt[2 * b + 1];
  }
  int used = 0;
  std::vector<std::pair<double, int>> rem;
  std::vector<double> ideal(2 * n_req, 0.0);
  for (int x = 0; x < 2 * n_req; ++x) {
    if (cap[x] == 0) continue;
    ideal[x] = W > 0 ? U * wgt[x] / W : 0.0;
    cnt[x] = std::min(cap[x], std::max(1, (int)std::floor(ideal[x])));
    used += cnt[x];
    if (cnt[x] < cap[x]) rem.push_back({ideal[x] - std::floor(ideal[x]), x});
  }
  // the one-unit minimum of small segments can overshoot the budget: take units
  // back from the most over-allocated segments (U >= min_units, so this ends)
  while (used > U) {
    int best = -1;
    double over = -1e300;
    for (int x = 0; x < 2 * n_req; ++x)
      if (cnt[x] > 1 && cnt[x] - ideal[x] > over) {
        over = cnt[x] - ideal[x];
        best = x;
      }
    if (best < 0) break;
    cnt[best] -= 1;
    used -= 1;
  }
  std::sort(rem.begin(), rem.end(), [](const std::pair<double, int>& a, const std::pair<double, int>& c) {
    return a.first > c.first || (a.first == c.first && a.second < c.second);
  });
  for (size_t k = 0; used < U && k < rem.size(); ++k) {
    cnt[rem[k].second] += 1;
    used += 1;
  }
  for (int b = 0; b < n_req; ++b)
    if (cnt[2 * b] > 32767 || cnt[2 * b + 1] > 32767) return fail(TPK_ERR_UNSUPPORTED, "request %d: too many splits", b);
  if (used * H > kMaxUnits) return fail(TPK_ERR_UNSUPPORTED, "could not plan within %d units", kMaxUnits);
  return TPK_OK;
}

// Timing events recorded around every decode-kernel launch while set (see
// tpk_set_decode_timing_events); external records, so that a captured graph
// records them on each replay.
cudaEvent_t g_decode_ev[2] = {nullptr, nullptr};

tpk_status launch_decode(const tpk_shape* s, const DecodeParams& p, const ReqPlan* req, cudaStream_t st) {
  if (g_decode_ev[0]) {
    cudaError_t e = cudaEventRecordWithFlags(g_decode_ev[0], st, cudaEventRecordExternal);
    if (e != cudaSuccess) return cuda_fail(e, "timing event");
  }
  cudaError_t e = use_simt(s) ? launch_decode_simt(p, req, st) : launch_decode_mma(p, req, st);
  if (e != cudaSuccess) return cuda_fail(e, "decode launch");
  if (g_decode_ev[1]) {
    e = cudaEventRecordWithFlags(g_decode_ev[1], st, cudaEventRecordExternal);
    if (e != cudaSuccess) return cuda_fail(e, "timing event");
  }
  return TPK_OK;
}

}  // namespace

void tpk::set_error(const char* msg) { g_err = msg; }

extern "C" {

const char* tpk_version(void) { return "tpk 0.1 (sm_103a)"; }

const char* tpk_last_error_string(void) { return g_err.c_str(); }

static tpk_status quantize_common(const tpk_shape* shape, const void* k_pool, const void* v_pool,
                                  const int32_t* src_slots, const int32_t* dst_slots, int n_pages,
                                  const float* ks_chan, const float* ks_tok, const float* vs_chan, void* rec_pool,
                                  tpk_stream_t stream) {
  tpk_status st = check_shape(shape);
  if (st != TPK_OK) return st;
  if (n_pages < 0) return fail(TPK_ERR_INVALID, "n_pages %d < 0", n_pages);
  if (n_pages == 0) return TPK_OK;
  if (!k_pool || !v_pool || !src_slots || !dst_slots || !rec_pool)
    return fail(TPK_ERR_INVALID, "null pointer argument");
  if (!aligned16(k_pool) || !aligned16(v_pool) || !aligned16(rec_pool))
    return fail(TPK_ERR_INVALID, "pools must be 16-byte aligned");
  if ((int64_t)n_pages * shape->kv_heads > 0x7fffffffLL) return fail(TPK_ERR_INVALID, "too many pages");
  int* status = status_ptr();
  if (!status) return fail(TPK_ERR_CUDA, "cannot resolve the device status word");
  QuantParams p;
  p.k_pool = static_cast<const uint16_t*>(k_pool);
  p.v_pool = static_cast<const uint16_t*>(v_pool);
  p.src = src_slots;
  p.dst = dst_slots;
  p.rec_pool = static_cast<uint8_t*>(rec_pool);
  p.g_kchan = ks_chan;
  p.g_ktok = ks_tok;
  p.g_vchan = vs_chan;
  p.kv_slots = shape->kv_slots;
  p.rec_slots = shape->rec_slots;
  p.status = status;
  p.H = shape->kv_heads;
  cudaError_t e = launch_quantize(p, n_pages, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "quantize launch");
  return TPK_OK;
}

tpk_status tpk_kv_quantize_pages(const tpk_shape* shape, const void* k_pool, const void* v_pool,
                                 const int32_t* src_slots, const int32_t* dst_slots, int n_pages, void* rec_pool,
                                 tpk_stream_t stream) {
  return quantize_common(shape, k_pool, v_pool, src_slots, dst_slots, n_pages, nullptr, nullptr, nullptr,
                         rec_pool, stream);
}

tpk_status tpk_kv_quantize_pages_given_scales(const tpk_shape* shape, const void* k_pool, const void* v_pool,
                                              const int32_t* src_slots, const int32_t* dst_slots, int n_pages,
                                              const float* ks_chan, const float* ks_tok, const float* vs_chan,
                                              void* rec_pool, tpk_stream_t stream) {
  if (n_pages > 0 && (!ks_chan || !ks_tok || !vs_chan)) return fail(TPK_ERR_INVALID, "null scale array");
  return quantize_common(shape, k_pool, v_pool, src_slots, dst_slots, n_pages, ks_chan, ks_tok, vs_chan,
                         rec_pool, stream);
}

tpk_status tpk_decode_attn_exact(const tpk_shape* shape, const void* q, const void* k_pool, const void* v_pool,
                                 const int32_t* page_table, int tok_begin, int tok_end, int num_splits,
                                 float* o_part, float* lse_part, tpk_stream_t stream) {
  tpk_status st = check_shape(shape);
  if (st != TPK_OK) return st;
  if (tok_begin < 0 || tok_end < tok_begin) return fail(TPK_ERR_INVALID, "bad token range [%d, %d)", tok_begin, tok_end);
  if (num_splits < 1 || num_splits > kMaxSplits) return fail(TPK_ERR_INVALID, "num_splits %d out of [1, %d]", num_splits, kMaxSplits);
  if (!q || !o_part || !lse_part) return fail(TPK_ERR_INVALID, "null pointer argument");
  if (tok_end > tok_begin && (!k_pool || !v_pool || !page_table)) return fail(TPK_ERR_INVALID, "null pool or page table");
  if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(o_part))
    return fail(TPK_ERR_INVALID, "q, pools and o_part must be 16-byte aligned");
  if ((int64_t)num_splits * shape->kv_heads > 0x7fffffffLL) return fail(TPK_ERR_INVALID, "grid too large");
  DecodeParams p;
  fill_common(p, shape, q);
  p.k_pool = static_cast<const uint16_t*>(k_pool);
  p.v_pool = static_cast<const uint16_t*>(v_pool);
  p.page_table = page_table;
  p.part_o = o_part;
  p.part_lse = lse_part;
  p.status = status_ptr();
  if (!p.status) return fail(TPK_ERR_CUDA, "cannot resolve the device status word");
  p.mode = kModePrimitive;
  p.n_req = 1;
  ReqPlan req = ReqPlan{0, 0, tok_begin, tok_end, 0, 0, 0, (int16_t)0, (int16_t)0};
  // int16 split counts: fold larger counts through the unit decode's int arithmetic
  if (num_splits > 32767) return fail(TPK_ERR_INVALID, "num_splits too large");
  req.splits_e = (int16_t)num_splits;
  p.n_units = num_splits * shape->kv_heads;
  if (tok_end > tok_begin) {
    st = make_pool_maps(p, shape, k_pool, v_pool);
    if (st != TPK_OK) return st;
  }
  return launch_decode(shape, p, &req, reinterpret_cast<cudaStream_t>(stream));
}

tpk_status tpk_decode_attn_int8(const tpk_shape* shape, const void* q, const void* rec_pool,
                                const int32_t* page_table8, int page_begin, int page_end, int num_splits,
                                float* o_part, float* lse_part, tpk_stream_t stream) {
  tpk_status st = check_shape(shape);
  if (st != TPK_OK) return st;
  if (page_begin < 0 || page_end < page_begin) return fail(TPK_ERR_INVALID, "bad page range [%d, %d)", page_begin, page_end);
  if (page_end > 0x7fffffff / kPageTokens) return fail(TPK_ERR_INVALID, "page range too large");
  if (num_splits < 1 || num_splits > kMaxSplits) return fail(TPK_ERR_INVALID, "num_splits %d out of [1, %d]", num_splits, kMaxSplits);
  if (!q || !o_part || !lse_part) return fail(TPK_ERR_INVALID, "null pointer argument");
  if (page_end > page_begin && (!rec_pool || !page_table8)) return fail(TPK_ERR_INVALID, "null pool or page table");
  if (!aligned16(q) || !aligned16(rec_pool) || !aligned16(o_part))
    return fail(TPK_ERR_INVALID, "q, rec_pool and o_part must be 16-byte aligned");
  DecodeParams p;
  fill_common(p, shape, q);
  p.rec_pool = static_cast<const uint8_t*>(rec_pool);
  p.page_table8 = page_table8;
  p.part_o = o_part;
  p.part_lse = lse_part;
  p.status = status_ptr();
  if (!p.status) return fail(TPK_ERR_CUDA, "cannot resolve the device status word");
  p.mode = kModePrimitive;
  p.n_req = 1;
  const ReqPlan req = ReqPlan{0, 0, 0, 0, 0, page_begin, page_end, (int16_t)0, (int16_t)num_splits};
  p.n_units = num_splits * shape->kv_heads;
  return launch_decode(shape, p, &req, reinterpret_cast<cudaStream_t>(stream));
}

tpk_status tpk_merge_lse(int n_parts, int rows, int head_dim, const float* o_parts, const float* lse_parts,
                         float* o_acc, float* lse_acc, tpk_stream_t stream) {
  if (head_dim != kHeadDim) return fail(TPK_ERR_UNSUPPORTED, "head_dim %d (only 256 supported)", head_dim);
  if (n_parts < 0 || rows < 0) return fail(TPK_ERR_INVALID, "negative n_parts or rows");
  if (rows == 0) return TPK_OK;
  if (!o_acc || !lse_acc || (n_parts > 0 && (!o_parts || !lse_parts)))
    return fail(TPK_ERR_INVALID, "null pointer argument");
  cudaError_t e = launch_merge(n_parts, rows, o_parts, lse_parts, o_acc, lse_acc,
                               reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "merge launch");
  return TPK_OK;
}

static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

size_t tpk_hybrid_workspace_bytes(const tpk_shape* shape, int n_req) {
  if (!shape || n_req < 1 || shape->kv_heads < 1) return 0;
  return align256((size_t)kMaxUnits * kGroup * 4) + (size_t)kMaxUnits * kGroup * kHeadDim * 4;
}

tpk_status tpk_workspace_init(void* ws, size_t ws_bytes, tpk_stream_t stream) {
  if (!ws) return fail(TPK_ERR_INVALID, "null workspace");
  cudaError_t e = cudaMemsetAsync(ws, 0, ws_bytes, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "workspace memset");
  return TPK_OK;
}

tpk_status tpk_decode_hybrid_batched(const tpk_shape* shape, int n_req, const void* q, const void* k_pool,
                                     const void* v_pool, const void* rec_pool, const int32_t* page_table,
                                     const int32_t* req_page_off, const int32_t* n_exact_tokens,
                                     const int32_t* page_table8, const int32_t* req_page_off8,
                                     const int32_t* n_int8_pages, float* o, float* lse, void* ws, size_t ws_bytes,
                                     tpk_stream_t stream) {
  tpk_status st = check_shape(shape);
  if (st != TPK_OK) return st;
  if (n_req < 1 || n_req > kMaxReqPerLaunch) return fail(TPK_ERR_INVALID, "n_req %d out of [1, %d]", n_req, kMaxReqPerLaunch);
  if (!q || !o || !lse || !ws || !req_page_off || !n_exact_tokens || !req_page_off8 || !n_int8_pages)
    return fail(TPK_ERR_INVALID, "null pointer argument");
  if (!aligned16(q) || !aligned16(o) || !aligned16(ws) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(rec_pool))
    return fail(TPK_ERR_INVALID, "device buffers must be 16-byte aligned");
  const int H = shape->kv_heads;
  size_t need = tpk_hybrid_workspace_bytes(shape, n_req);
  if (ws_bytes < need) return fail(TPK_ERR_NOMEM, "workspace %zu bytes < %zu required", ws_bytes, need);
  // ---- validate the host metadata and measure the work
  double total = 0.0;
  bool any_e = false, any_8 = false;
  for (int b = 0; b < n_req; ++b) {
    int ne = n_exact_tokens[b], n8 = n_int8_pages[b];
    if (ne < 0 || n8 < 0) return fail(TPK_ERR_INVALID, "request %d: negative length", b);
    if (n8 > 0x7fffffff / kPageTokens) return fail(TPK_ERR_INVALID, "request %d: too many pages", b);
    int have_e = req_page_off[b + 1] - req_page_off[b];
    int have_8 = req_page_off8[b + 1] - req_page_off8[b];
    if (req_page_off[b] < 0 || have_e < (ne + kPageTokens - 1) / kPageTokens)
      return fail(TPK_ERR_INVALID, "request %d: exact page table holds %d pages, %d tokens need %d", b, have_e, ne,
                  (ne + kPageTokens - 1) / kPageTokens);
    if (req_page_off8[b] < 0 || have_8 < n8)
      return fail(TPK_ERR_INVALID, "request %d: 8-bit page table holds %d pages, need %d", b, have_8, n8);
    any_e |= ne > 0;
    any_8 |= n8 > 0;
    total += (double)H * (1024.0 * ne + (double)kRecordBytes * n8);
  }
  if (any_e && (!k_pool || !v_pool || !page_table)) return fail(TPK_ERR_INVALID, "null BF16 pool or page table");
  if (any_8 && (!rec_pool || !page_table8)) return fail(TPK_ERR_INVALID, "null 8-bit pool or page table");
  std::vector<int> cnt;
  st = plan_splits(H, n_req, n_exact_tokens, n_int8_pages, num_sms() * blocks_per_sm(shape), cnt);
  if (st != TPK_OK) return st;
  DecodeParams p;
  fill_common(p, shape, q);
  std::vector<ReqPlan> req(n_req);
  int units = 0;
  for (int b = 0; b < n_req; ++b) {
    const int se = cnt[2 * b], s8 = cnt[2 * b + 1];
    req[b] = ReqPlan{units, req_page_off[b], 0, n_exact_tokens[b], req_page_off8[b], 0, n_int8_pages[b],
                       (int16_t)se, (int16_t)s8};
    units += H * (se + s8);
  }
  if (units > kMaxUnits) return fail(TPK_ERR_UNSUPPORTED, "could not plan within %d units", kMaxUnits);
  p.n_units = units;
  p.k_pool = static_cast<const uint16_t*>(k_pool);
  p.v_pool = static_cast<const uint16_t*>(v_pool);
  p.rec_pool = static_cast<const uint8_t*>(rec_pool);
  p.page_table = page_table;
  p.page_table8 = page_table8;
  uint8_t* w = static_cast<uint8_t*>(ws);
  p.part_lse = reinterpret_cast<float*>(w);
  w += align256((size_t)kMaxUnits * kGroup * 4);
  p.part_o = reinterpret_cast<float*>(w);
  p.out_o = o;
  p.out_lse = lse;
  p.mode = kModeFold;
  p.n_req = n_req;
  p.status = status_ptr();
  if (!p.status) return fail(TPK_ERR_CUDA, "cannot resolve the device status word");
  if (any_e) {
    st = make_pool_maps(p, shape, k_pool, v_pool);
    if (st != TPK_OK) return st;
  }
  st = launch_decode(shape, p, req.data(), reinterpret_cast<cudaStream_t>(stream));
  if (st != TPK_OK) return st;
  bool any_split = false;
  for (int b = 0; b < n_req; ++b) any_split |= req[b].splits_e + req[b].splits_8 > 1;
  if (any_split) {
    cudaError_t e = launch_fold(p, req.data(), reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "fold launch");
  }
  return TPK_OK;
}

tpk_status tpk_set_decode_timing_events(void* before, void* after) {
  if ((before == nullptr) != (after == nullptr)) return fail(TPK_ERR_INVALID, "set both timing events or neither");
  g_decode_ev[0] = static_cast<cudaEvent_t>(before);
  g_decode_ev[1] = static_cast<cudaEvent_t>(after);
  return TPK_OK;
}

tpk_status tpk_set_test_wait(uint64_t wait_limit_ns, int stall_unit) {
  if (stall_unit < -1) return fail(TPK_ERR_INVALID, "stall_unit %d < -1", stall_unit);
  if (wait_limit_ns > 60000000000ull) return fail(TPK_ERR_INVALID, "wait limit above 60 s");
  g_test_wait_ns.store(wait_limit_ns, std::memory_order_relaxed);
  g_test_stall_unit.store(stall_unit, std::memory_order_relaxed);
  return TPK_OK;
}

tpk_status tpk_hybrid_plan(const tpk_shape* shape, int n_req, const int32_t* n_exact_tokens,
                           const int32_t* n_int8_pages, int resident_blocks, int32_t* splits_exact,
                           int32_t* splits_int8, int32_t* n_units) {
  tpk_status st = check_shape(shape);
  if (st != TPK_OK) return st;
  if (n_req < 1 || n_req > kMaxReqPerLaunch) return fail(TPK_ERR_INVALID, "n_req %d out of [1, %d]", n_req, kMaxReqPerLaunch);
  if (!n_exact_tokens || !n_int8_pages || !splits_exact || !splits_int8 || !n_units)
    return fail(TPK_ERR_INVALID, "null pointer argument");
  if (resident_blocks < 0) return fail(TPK_ERR_INVALID, "resident_blocks %d < 0", resident_blocks);
  for (int b = 0; b < n_req; ++b) {
    if (n_exact_tokens[b] < 0 || n_int8_pages[b] < 0) return fail(TPK_ERR_INVALID, "request %d: negative length", b);
    if (n_int8_pages[b] > 0x7fffffff / kPageTokens) return fail(TPK_ERR_INVALID, "request %d: too many pages", b);
  }
  const int per_wave = resident_blocks > 0 ? resident_blocks : num_sms() * blocks_per_sm(shape);
  std::vector<int> cnt;
  st = plan_splits(shape->kv_heads, n_req, n_exact_tokens, n_int8_pages, per_wave, cnt);
  if (st != TPK_OK) return st;
  int units = 0;
  for (int b = 0; b < n_req; ++b) {
    splits_exact[b] = cnt[2 * b];
    splits_int8[b] = cnt[2 * b + 1];
    units += shape->kv_heads * (cnt[2 * b] + cnt[2 * b + 1]);
  }
  *n_units = units;
  return TPK_OK;
}

tpk_status tpk_get_device_status(int* flags, int reset, tpk_stream_t stream) {
  if (!flags) return fail(TPK_ERR_INVALID, "null flags");
  int* d = status_ptr();
  if (!d) return fail(TPK_ERR_CUDA, "cannot resolve the device status word");
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
  e = cudaMemcpy(flags, d, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "status read");
  if (reset) {
    e = cudaMemset(d, 0, sizeof(int));
    if (e != cudaSuccess) return cuda_fail(e, "status reset");
  }
  if (*flags & kStatusTimeout) return fail(TPK_ERR_TIMEOUT, "a device-side wait gave up (status %d)", *flags);
  if (*flags & kStatusBadSlot) return fail(TPK_ERR_BOUNDS, "a page-table entry outside the pool was skipped");
  if (*flags & kStatusBadRecord) return fail(TPK_ERR_FORMAT, "a malformed 13-bit record was skipped");
  return TPK_OK;
}

tpk_status tpk_kv_pack13_pages(const tpk_shape* shape, const void* k_pool, const void* v_pool,
                               const int32_t* src_slots, const int32_t* dst_slots, int n_pages, void* pack_pool,
                               int64_t pack_slots, tpk_stream_t stream) {
  tpk_status st = check_shape(shape);
  if (st != TPK_OK) return st;
  if (n_pages < 0) return fail(TPK_ERR_INVALID, "n_pages %d < 0", n_pages);
  if (pack_slots < 0) return fail(TPK_ERR_INVALID, "pack_slots %lld < 0", (long long)pack_slots);
  if (n_pages == 0) return TPK_OK;
  if (!k_pool || !v_pool || !src_slots || !dst_slots || !pack_pool) return fail(TPK_ERR_INVALID, "null pointer argument");
  if (!aligned16(k_pool) || !aligned16(v_pool) || !aligned16(pack_pool))
    return fail(TPK_ERR_INVALID, "pools must be 16-byte aligned");
  if ((int64_t)n_pages * shape->kv_heads > 0x7fffffffLL) return fail(TPK_ERR_INVALID, "too many pages");
  int* status = status_ptr();
  if (!status) return fail(TPK_ERR_CUDA, "cannot resolve the device status word");
  Pack13Params p;
  p.k_pool = static_cast<const uint16_t*>(k_pool);
  p.v_pool = static_cast<const uint16_t*>(v_pool);
  p.src = src_slots;
  p.dst = dst_slots;
  p.out = static_cast<uint8_t*>(pack_pool);
  p.kv_slots = shape->kv_slots;
  p.out_slots = pack_slots;
  p.status = status;
  p.H = shape->kv_heads;
  cudaError_t e = launch_pack13(p, n_pages, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "pack13 launch");
  return TPK_OK;
}

tpk_status tpk_kv_unpack13_pages(const tpk_shape* shape, const void* src, int64_t src_bytes,
                                 const int64_t* rec_offsets, const int32_t* dst_slots, int n_pages, void* k_pool,
                                 void* v_pool, tpk_stream_t stream) {
  tpk_status st = check_shape(shape);
  if (st != TPK_OK) return st;
  if (n_pages < 0) return fail(TPK_ERR_INVALID, "n_pages %d < 0", n_pages);
  if (src_bytes < 0) return fail(TPK_ERR_INVALID, "src_bytes %lld < 0", (long long)src_bytes);
  if (n_pages == 0) return TPK_OK;
  if (!src || !rec_offsets || !dst_slots || !k_pool || !v_pool) return fail(TPK_ERR_INVALID, "null pointer argument");
  if (!aligned16(src) || !aligned16(k_pool) || !aligned16(v_pool))
    return fail(TPK_ERR_INVALID, "src and pools must be 16-byte aligned");
  if ((int64_t)n_pages * shape->kv_heads > 0x7fffffffLL) return fail(TPK_ERR_INVALID, "too many pages");
  int* status = status_ptr();
  if (!status) return fail(TPK_ERR_CUDA, "cannot resolve the device status word");
  Unpack13Params p;
  p.src = static_cast<const uint8_t*>(src);
  p.offsets = rec_offsets;
  p.src_bytes = src_bytes;
  p.dst = dst_slots;
  p.k_pool = static_cast<uint16_t*>(k_pool);
  p.v_pool = static_cast<uint16_t*>(v_pool);
  p.kv_slots = shape->kv_slots;
  p.status = status;
  p.H = shape->kv_heads;
  cudaError_t e = launch_unpack13(p, n_pages, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "unpack13 launch");
  return TPK_OK;
}

}  // extern "C"
