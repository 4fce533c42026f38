// Multi-request hybrid decode without a caller-provided workspace.
//
// Some callers cannot give the library device memory for its scratch: a plugin
// inside a host engine that owns every device allocation through its own pool
// and offers plugins no way to request more, or a runtime with a fixed,
// pre-reserved memory budget that must not grow once serving has started.  For
// them this entry point keeps the scratch (the split units' partial results) in
// a file-scope device array that every GPU loading the library holds until the
// process exits.  It allocates nothing: no cudaMalloc, no cudaFree, no
// allocating library call.
#include <cuda_runtime.h>

#include <mutex>

#include "tpk.h"

namespace tpk {
void set_error(const char* msg);  // api.cu: sets the message tpk_last_error_string returns
}

namespace {

// Fixed scratch: room for the largest split plan the multi-request call makes
// (2048 units x 8 rows x (256 + 1) floats).
constexpr size_t kStaticScratchBytes = 16842752;
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices] = {nullptr};
std::mutex g_setup_lock;

// Device address of the scratch array on the current device, resolved once per
// device.  In host code the array's name is only a stand-in for the device
// symbol, so its address must come from cudaGetSymbolAddress.
void* scratch_on_current_device(tpk_status* st) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    *st = TPK_ERR_CUDA;
    tpk::set_error("no usable current device for the static scratch");
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_setup_lock);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess || !p) {
      *st = TPK_ERR_CUDA;
      tpk::set_error("cudaGetSymbolAddress failed for the static scratch");
      return nullptr;
    }
    g_scratch_ptr[dev] = p;
  }
  *st = TPK_OK;
  return g_scratch_ptr[dev];
}

}  // namespace

extern "C" size_t tpk_static_scratch_bytes(void) { return kStaticScratchBytes; }

extern "C" tpk_status tpk_decode_hybrid_batched_static(const tpk_shape* shape, int n_req, const void* q,
                                                       const void* k_pool, const void* v_pool, const void* rec_pool,
                                                       const int32_t* page_table, const int32_t* req_page_off,
                                                       const int32_t* n_exact_tokens, const int32_t* page_table8,
                                                       const int32_t* req_page_off8, const int32_t* n_int8_pages,
                                                       float* o, float* lse, tpk_stream_t stream) {
  const size_t need = tpk_hybrid_workspace_bytes(shape, n_req);
  if (need == 0) {
    tpk::set_error("invalid shape or n_req");
    return TPK_ERR_INVALID;
  }
  if (need > kStaticScratchBytes) {
    tpk::set_error("this call needs more scratch than the static array holds");
    return TPK_ERR_NOMEM;
  }
  tpk_status st;
  void* scratch = scratch_on_current_device(&st);
  if (!scratch) return st;
  return tpk_decode_hybrid_batched(shape, n_req, q, k_pool, v_pool, rec_pool, page_table, req_page_off,
                                   n_exact_tokens, page_table8, req_page_off8, n_int8_pages, o, lse, scratch,
                                   kStaticScratchBytes, stream);
}
