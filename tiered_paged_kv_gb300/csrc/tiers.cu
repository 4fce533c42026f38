// Incremental page conversion and publication during decode.
//
// A tier manager follows the histories of n_req requests across n_layers
// attention layers that share one page table per request (page p of a request
// sits in the same slot of every layer's pools).  Every step it (1) publishes
// the pages whose conversion has finished in every layer -- they move from the
// exact tier to the 8-bit tier, in all layers at once, because the layers share
// the tables -- (2) starts, on the caller's conversion stream, the conversion in
// every layer of each whole page that is older than the recent window and has
// been written by every layer, and (3) uploads the step's two page tables (in the
// decode stream's order) for the multi-request decode call.  A page is served
// exact until the event recorded after all its layers' conversions has
// completed, so no decode reads a half-written record; the swap from one tier to
// the other happens between steps, through the page tables ("ActiveKV":
// compressed history converted in the background and published to the decoder;
// "model quantization", "An 8-bit page format shaped for its kernel": conversion
// only for pages fully written in every layer, served exact until published).
//
// Host-authoritative history ("ActiveKV", "The idea": host memory holds the
// authoritative copy, the GPU the slices a step needs): when pinned host record
// pools are given, each converted record is also copied into its layer's host
// pool before the conversion's event, so a published page's records are in the
// host image too, ready to be staged.
//
// Record slot of a page = its BF16 slot (the record pool is indexed like the KV
// pools).  All device and pinned host buffers are allocated once, at creation.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <deque>
#include <vector>

#include "tpk.h"

namespace tpk {
void set_error(const char* msg);  // api.cu: sets the message tpk_last_error_string returns
}

namespace {

tpk_status tfail(tpk_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  tpk::set_error(buf);
  return s;
}

tpk_status tcuda(cudaError_t e, const char* what) { return tfail(TPK_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e)); }

constexpr int kPage = 64;

struct Request {
  int n_tokens = 0;
  std::vector<int32_t> slots;  // BF16 slot of each logical page (the same in every layer)
  std::vector<int> written;    // tokens each layer has written
  int published = 0;           // pages [0, published) are served from records
  int converting = 0;          // pages [published, published + converting) are being converted
};

struct Conversion {
  cudaEvent_t done;
  int b, count;
};

}  // namespace

struct tpk_tiers {
  tpk_shape shape;
  int device = 0;
  int n_req = 0, max_pages = 0, recent = 0, n_layers = 1;
  std::vector<const void*> k_pool, v_pool;  // per layer (device)
  std::vector<void*> rec_pool;              // per layer (device)
  std::vector<void*> host_rec;              // per layer (pinned host), or empty
  std::vector<Request> req;
  std::deque<Conversion> inflight;
  std::vector<cudaEvent_t> spare_events;
  // device: conversion slot lists (ring) and two page-table buffers
  int32_t* d_conv = nullptr;  // [conv_cap]
  int conv_cap = 0, conv_head = 0;
  int32_t* d_pt[2] = {nullptr, nullptr};   // [n_req * max_pages] each
  int32_t* d_pt8[2] = {nullptr, nullptr};
  // pinned host staging of the uploads (two generations) and their events
  int32_t* h_stage[2] = {nullptr, nullptr};  // [2 * n_req * max_pages + conv_cap]
  cudaEvent_t stage_done[2] = {nullptr, nullptr};       // decode stream: table uploads done
  cudaEvent_t stage_conv_done[2] = {nullptr, nullptr};  // conversion stream: slot upload done
  bool stage_used[2] = {false, false};
  bool stage_conv_used[2] = {false, false};
  cudaEvent_t order = nullptr;  // the decode stream's position, for the conversion stream to wait on
  int gen = 0;
  // the plan handed back to the caller (host arrays live here)
  std::vector<int32_t> off, off8, n_ex, n8;
  // the tables last uploaded (and into which generation), to skip unchanged uploads
  std::vector<int32_t> last_pt, last_pt8;
  int last_gen = -1;
  long long published_total = 0, started_total = 0;
};

extern "C" {

size_t tpk_tiers_device_bytes(int n_req, int max_pages) {
  if (n_req < 1 || max_pages < 1) return 0;
  const size_t pt = (size_t)n_req * max_pages * sizeof(int32_t);
  const size_t conv = (size_t)4 * n_req * max_pages * sizeof(int32_t);
  return 4 * ((pt + 255) & ~size_t(255)) + ((conv + 255) & ~size_t(255));
}

tpk_status tpk_tiers_create_layers(const tpk_shape* shape, int n_layers, int n_req, int max_pages, int recent_tokens,
                                   const void* const* k_pools, const void* const* v_pools, void* const* rec_pools,
                                   void* const* host_rec_pools, void* dev_scratch, size_t dev_scratch_bytes,
                                   tpk_tiers** out) {
  if (!out) return tfail(TPK_ERR_INVALID, "null output pointer");
  *out = nullptr;
  if (!shape || shape->kv_heads < 1) return tfail(TPK_ERR_INVALID, "bad shape");
  if (shape->group != 8 || shape->head_dim != 256 || shape->page_tokens != kPage)
    return tfail(TPK_ERR_UNSUPPORTED, "only group 8, head_dim 256, 64-token pages");
  if (n_layers < 1 || n_layers > 1024) return tfail(TPK_ERR_INVALID, "n_layers %d out of [1, 1024]", n_layers);
  if (n_req < 1 || max_pages < 1) return tfail(TPK_ERR_INVALID, "n_req %d, max_pages %d", n_req, max_pages);
  if (recent_tokens < 0) return tfail(TPK_ERR_INVALID, "recent_tokens %d < 0", recent_tokens);
  if (!k_pools || !v_pools || !rec_pools) return tfail(TPK_ERR_INVALID, "null pool array");
  for (int l = 0; l < n_layers; ++l) {
    if (!k_pools[l] || !v_pools[l] || !rec_pools[l]) return tfail(TPK_ERR_INVALID, "layer %d: null pool", l);
    if (host_rec_pools) {
      if (!host_rec_pools[l]) return tfail(TPK_ERR_INVALID, "layer %d: null host record pool", l);
      cudaPointerAttributes a;
      cudaError_t e = cudaPointerGetAttributes(&a, host_rec_pools[l]);
      if (e != cudaSuccess) return tcuda(e, "cudaPointerGetAttributes (host record pool)");
      if (a.type != cudaMemoryTypeHost)
        return tfail(TPK_ERR_INVALID, "layer %d: the host record pool is not pinned host memory", l);
    }
  }
  const size_t need = tpk_tiers_device_bytes(n_req, max_pages);
  if (!dev_scratch || dev_scratch_bytes < need)
    return tfail(TPK_ERR_NOMEM, "device scratch %zu bytes < %zu required", dev_scratch_bytes, need);
  if (reinterpret_cast<uintptr_t>(dev_scratch) & 255u) return tfail(TPK_ERR_INVALID, "device scratch not 256-byte aligned");
  tpk_tiers* t = new tpk_tiers;
  t->shape = *shape;
  t->n_req = n_req;
  t->max_pages = max_pages;
  t->recent = recent_tokens;
  t->n_layers = n_layers;
  t->k_pool.assign(k_pools, k_pools + n_layers);
  t->v_pool.assign(v_pools, v_pools + n_layers);
  t->rec_pool.assign(rec_pools, rec_pools + n_layers);
  if (host_rec_pools) t->host_rec.assign(host_rec_pools, host_rec_pools + n_layers);
  t->req.resize(n_req);
  for (auto& r : t->req) r.written.assign(n_layers, 0);
  cudaGetDevice(&t->device);
  const size_t pt = (((size_t)n_req * max_pages * sizeof(int32_t)) + 255) & ~size_t(255);
  char* base = static_cast<char*>(dev_scratch);
  for (int g = 0; g < 2; ++g) {
    t->d_pt[g] = reinterpret_cast<int32_t*>(base + (2 * g) * pt);
    t->d_pt8[g] = reinterpret_cast<int32_t*>(base + (2 * g + 1) * pt);
  }
  t->d_conv = reinterpret_cast<int32_t*>(base + 4 * pt);
  t->conv_cap = 4 * n_req * max_pages;
  cudaError_t e = cudaSuccess;
  const size_t stage_words = (size_t)2 * n_req * max_pages + t->conv_cap;
  for (int g = 0; g < 2 && e == cudaSuccess; ++g) {
    void* h = nullptr;
    e = cudaHostAlloc(&h, stage_words * sizeof(int32_t), cudaHostAllocDefault);
    t->h_stage[g] = static_cast<int32_t*>(h);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&t->stage_done[g], cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&t->stage_conv_done[g], cudaEventDisableTiming);
  }
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&t->order, cudaEventDisableTiming);
  if (e != cudaSuccess) {
    for (int g = 0; g < 2; ++g) {
      if (t->h_stage[g]) cudaFreeHost(t->h_stage[g]);
      if (t->stage_done[g]) cudaEventDestroy(t->stage_done[g]);
      if (t->stage_conv_done[g]) cudaEventDestroy(t->stage_conv_done[g]);
    }
    if (t->order) cudaEventDestroy(t->order);
    delete t;
    return tcuda(e, "tier manager staging");
  }
  t->off.assign(n_req + 1, 0);
  t->off8.assign(n_req + 1, 0);
  t->n_ex.assign(n_req, 0);
  t->n8.assign(n_req, 0);
  *out = t;
  return TPK_OK;
}

tpk_status tpk_tiers_create(const tpk_shape* shape, int n_req, int max_pages, int recent_tokens, const void* k_pool,
                            const void* v_pool, void* rec_pool, void* dev_scratch, size_t dev_scratch_bytes,
                            tpk_tiers** out) {
  return tpk_tiers_create_layers(shape, 1, n_req, max_pages, recent_tokens, &k_pool, &v_pool, &rec_pool, nullptr,
                                 dev_scratch, dev_scratch_bytes, out);
}

tpk_status tpk_tiers_update_layers(tpk_tiers* t, int b, int n_tokens, const int32_t* page_slots,
                                   const int32_t* layer_written) {
  if (!t) return tfail(TPK_ERR_INVALID, "null tier manager");
  if (b < 0 || b >= t->n_req) return tfail(TPK_ERR_INVALID, "request %d out of [0, %d)", b, t->n_req);
  Request& r = t->req[b];
  if (n_tokens < r.n_tokens) return tfail(TPK_ERR_INVALID, "request %d: history shrank (%d -> %d)", b, r.n_tokens, n_tokens);
  const int pages = (n_tokens + kPage - 1) / kPage;
  if (pages > t->max_pages) return tfail(TPK_ERR_INVALID, "request %d: %d pages > max_pages %d", b, pages, t->max_pages);
  if (pages > 0 && !page_slots) return tfail(TPK_ERR_INVALID, "null page slots");
  // pages already converted or being converted must keep their slots, and stay
  // written in every layer
  const int fixed = r.published + r.converting;
  for (int p = 0; p < fixed && p < pages; ++p)
    if (page_slots[p] != r.slots[p])
      return tfail(TPK_ERR_INVALID, "request %d: page %d moved while converted or being converted", b, p);
  if (layer_written)
    for (int l = 0; l < t->n_layers; ++l)
      if (layer_written[l] < kPage * fixed || layer_written[l] > n_tokens)
        return tfail(TPK_ERR_INVALID, "request %d, layer %d: %d tokens written, outside [%d, %d]", b, l,
                     layer_written[l], kPage * fixed, n_tokens);
  for (int p = 0; p < pages; ++p)
    if (page_slots[p] < 0 || (t->shape.kv_slots > 0 && page_slots[p] >= t->shape.kv_slots))
      return tfail(TPK_ERR_BOUNDS, "request %d: page %d slot %d outside the pool", b, p, page_slots[p]);
  r.slots.assign(page_slots, page_slots + pages);
  r.n_tokens = n_tokens;
  for (int l = 0; l < t->n_layers; ++l) r.written[l] = layer_written ? layer_written[l] : n_tokens;
  return TPK_OK;
}

tpk_status tpk_tiers_update(tpk_tiers* t, int b, int n_tokens, const int32_t* page_slots) {
  return tpk_tiers_update_layers(t, b, n_tokens, page_slots, nullptr);
}

// Publish finished conversions (in launch order), start new ones, upload the page
// tables.  Host arrays of the plan stay valid until the next call.
tpk_status tpk_tiers_step(tpk_tiers* t, tpk_stream_t conv_stream, tpk_stream_t decode_stream, tpk_tiers_plan* plan) {
  if (!t || !plan) return tfail(TPK_ERR_INVALID, "null argument");
  int dev = -1;
  cudaGetDevice(&dev);
  if (dev != t->device) return tfail(TPK_ERR_INVALID, "tier manager belongs to device %d", t->device);
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(conv_stream);
  cudaStream_t ds = reinterpret_cast<cudaStream_t>(decode_stream);
  // 1. publication: a conversion counts once its event has completed
  int published = 0;
  while (!t->inflight.empty()) {
    Conversion& c = t->inflight.front();
    cudaError_t q = cudaEventQuery(c.done);
    if (q == cudaErrorNotReady) break;
    if (q != cudaSuccess) return tcuda(q, "conversion event");
    Request& r = t->req[c.b];
    r.published += c.count;
    r.converting -= c.count;
    published += c.count;
    t->spare_events.push_back(c.done);
    t->inflight.pop_front();
  }
  // 2. pick the staging generation (its previous uploads must have been read)
  const int g = t->gen;
  t->gen ^= 1;
  {
    cudaError_t e = cudaSuccess;
    if (t->stage_used[g]) e = cudaEventSynchronize(t->stage_done[g]);
    if (e == cudaSuccess && t->stage_conv_used[g]) e = cudaEventSynchronize(t->stage_conv_done[g]);
    if (e != cudaSuccess) return tcuda(e, "staging reuse");
  }
  t->stage_used[g] = false;
  t->stage_conv_used[g] = false;
  int32_t* hs = t->h_stage[g];
  const size_t table_words = (size_t)t->n_req * t->max_pages;
  int32_t* h_pt = hs;
  int32_t* h_pt8 = hs + table_words;
  int32_t* h_conv = hs + 2 * table_words;
  // 3. new conversions: whole pages older than the recent window and written by
  //    every layer
  int n_conv = 0;
  int started = 0;
  std::vector<std::pair<int, int>> batch;  // (request, count), in the order of h_conv
  for (int b = 0; b < t->n_req; ++b) {
    Request& r = t->req[b];
    int eligible = r.n_tokens > t->recent ? (r.n_tokens - t->recent) / kPage : 0;
    for (int l = 0; l < t->n_layers; ++l) eligible = std::min(eligible, r.written[l] / kPage);
    const int first = r.published + r.converting;
    const int count = eligible - first;
    if (count <= 0) continue;
    if (n_conv + count > t->conv_cap) break;  // the rest waits for the next step
    for (int p = 0; p < count; ++p) h_conv[n_conv + p] = r.slots[first + p];
    batch.push_back({b, count});
    n_conv += count;
  }
  if (n_conv > 0) {
    // the conversion reads BF16 pages the decode stream's earlier work wrote
    cudaError_t e = cudaEventRecord(t->order, ds);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(cs, t->order, 0);
    if (e != cudaSuccess) return tcuda(e, "stream order");
    // (the slot ring is written and read on the conversion stream only, in order)
    if (t->conv_head + n_conv > t->conv_cap) t->conv_head = 0;
    int32_t* d = t->d_conv + t->conv_head;
    t->conv_head += n_conv;
    e = cudaMemcpyAsync(d, h_conv, n_conv * sizeof(int32_t), cudaMemcpyHostToDevice, cs);
    if (e == cudaSuccess) e = cudaEventRecord(t->stage_conv_done[g], cs);
    if (e != cudaSuccess) return tcuda(e, "conversion slot upload");
    t->stage_conv_used[g] = true;
    for (int l = 0; l < t->n_layers; ++l) {
      tpk_status st =
          tpk_kv_quantize_pages(&t->shape, t->k_pool[l], t->v_pool[l], d, d, n_conv, t->rec_pool[l], conv_stream);
      if (st != TPK_OK) return st;
    }
    // the host image gets every converted record before any of the events below
    // (runs of consecutive slots as one copy)
    if (!t->host_rec.empty()) {
      const size_t per_slot = (size_t)t->shape.kv_heads * TPK_RECORD_BYTES;
      for (int l = 0; l < t->n_layers; ++l)
        for (int i = 0; i < n_conv;) {
          int j = i + 1;
          while (j < n_conv && h_conv[j] == h_conv[j - 1] + 1) ++j;
          const size_t off = (size_t)h_conv[i] * per_slot;
          e = cudaMemcpyAsync(static_cast<char*>(t->host_rec[l]) + off, static_cast<const char*>(t->rec_pool[l]) + off,
                              (size_t)(j - i) * per_slot, cudaMemcpyDeviceToHost, cs);
          if (e != cudaSuccess) return tcuda(e, "record copy to the host image");
          i = j;
        }
    }
    for (const auto& bc : batch) {
      cudaEvent_t ev;
      if (!t->spare_events.empty()) {
        ev = t->spare_events.back();
        t->spare_events.pop_back();
      } else if ((e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming)) != cudaSuccess) {
        return tcuda(e, "conversion event");
      }
      e = cudaEventRecord(ev, cs);
      if (e != cudaSuccess) return tcuda(e, "conversion event record");
      t->inflight.push_back({ev, bc.first, bc.second});
      t->req[bc.first].converting += bc.second;
      started += bc.second;
    }
  }
  // 4. the step's page tables: 8-bit pages [0, published), exact pages after them
  //    (uploaded only when they differ from the last upload; otherwise the
  //    generation holding that upload is handed out again)
  int e_off = 0, p_off = 0;
  for (int b = 0; b < t->n_req; ++b) {
    const Request& r = t->req[b];
    const int pages = (int)r.slots.size();
    t->off[b] = e_off;
    t->off8[b] = p_off;
    for (int p = 0; p < r.published; ++p) h_pt8[p_off++] = r.slots[p];
    for (int p = r.published; p < pages; ++p) h_pt[e_off++] = r.slots[p];
    t->n8[b] = r.published;
    t->n_ex[b] = r.n_tokens - kPage * r.published;
  }
  t->off[t->n_req] = e_off;
  t->off8[t->n_req] = p_off;
  const bool same = t->last_gen >= 0 && (int)t->last_pt.size() == e_off && (int)t->last_pt8.size() == p_off &&
                    std::equal(t->last_pt.begin(), t->last_pt.end(), h_pt) &&
                    std::equal(t->last_pt8.begin(), t->last_pt8.end(), h_pt8);
  int tg = g;  // generation whose device tables this step uses
  if (same) {
    tg = t->last_gen;
    t->gen = g;  // this step's staging generation stays free for the next one
  } else {
    if (e_off > 0) {
      cudaError_t e = cudaMemcpyAsync(t->d_pt[g], h_pt, e_off * sizeof(int32_t), cudaMemcpyHostToDevice, ds);
      if (e != cudaSuccess) return tcuda(e, "page table upload");
    }
    if (p_off > 0) {
      cudaError_t e = cudaMemcpyAsync(t->d_pt8[g], h_pt8, p_off * sizeof(int32_t), cudaMemcpyHostToDevice, ds);
      if (e != cudaSuccess) return tcuda(e, "page table upload");
    }
    // this staging generation is reused two uploads later, once these copies are done
    cudaError_t e = cudaEventRecord(t->stage_done[g], ds);
    if (e != cudaSuccess) return tcuda(e, "staging event");
    t->stage_used[g] = true;
    t->last_pt.assign(h_pt, h_pt + e_off);
    t->last_pt8.assign(h_pt8, h_pt8 + p_off);
    t->last_gen = g;
  }
  t->published_total += published;
  t->started_total += started;
  plan->page_table = t->d_pt[tg];
  plan->req_page_off = t->off.data();
  plan->n_exact_tokens = t->n_ex.data();
  plan->page_table8 = t->d_pt8[tg];
  plan->req_page_off8 = t->off8.data();
  plan->n_int8_pages = t->n8.data();
  plan->pages_published = published;
  plan->pages_started = started;
  plan->pages_converting = 0;
  for (const auto& c : t->inflight) plan->pages_converting += c.count;
  return TPK_OK;
}

tpk_status tpk_tiers_sync(tpk_tiers* t) {
  if (!t) return tfail(TPK_ERR_INVALID, "null tier manager");
  for (const auto& c : t->inflight) {
    cudaError_t e = cudaEventSynchronize(c.done);
    if (e != cudaSuccess) return tcuda(e, "conversion event");
  }
  return TPK_OK;
}

tpk_status tpk_tiers_destroy(tpk_tiers* t) {
  if (!t) return TPK_OK;
  tpk_status st = tpk_tiers_sync(t);
  for (int g = 0; g < 2; ++g) {
    if (t->stage_used[g]) cudaEventSynchronize(t->stage_done[g]);
    if (t->stage_conv_used[g]) cudaEventSynchronize(t->stage_conv_done[g]);
    cudaEventDestroy(t->stage_done[g]);
    cudaEventDestroy(t->stage_conv_done[g]);
    cudaFreeHost(t->h_stage[g]);
  }
  cudaEventDestroy(t->order);
  for (auto& c : t->inflight) cudaEventDestroy(c.done);
  for (cudaEvent_t ev : t->spare_events) cudaEventDestroy(ev);
  delete t;
  return st;
}

}  // extern "C"
