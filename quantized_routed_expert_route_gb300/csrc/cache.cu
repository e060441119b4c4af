// Exact-geometry expert cache for expert banks larger than the GPU's memory.
//
// FreeToken issue #194, "avoid max-stride padding for heterogeneous GGUF
// expert banks", Proposed design: the byte-denominated bank arena is carved
// into disjoint exact-width pools, one per geometry (the tuple of row sizes),
// each with its own tags and LRU state; decode views and LRU updates are
// routed by layer; compact pinned-host rows are copied straight into the
// slots with no payload-sized device temporary.
//
// Here a pool is an ordinary bank over device memory whose "experts" are the
// slots (E = slots), so every decode path runs on it unchanged once a
// request's routing ids are remapped to slots.  moe_cache_acquire keeps the
// LRU state on the host: it maps each routed (layer, expert) to a slot,
// evicting the least recently used slot for each miss, and enqueues one copy
// per projection and miss from the layer's compact rows (any memory the
// device can read; pinned host memory for asynchronous copies) into the
// slot, plus the expert's scale row.  With exact-width slots the rows keep
// their compact layout, so each copy is a single contiguous transfer.  When
// the layer's rows live in memory the GPU addresses directly (pinned host
// memory, reached over the host link, or device memory), all of a request's
// copies run as one kernel in which every SM loads and stores 16-byte
// vectors; other sources go through the copy engine (cudaMemcpyAsync).
#include <cuda_runtime.h>

#include <cstring>
#include <new>
#include <unordered_map>
#include <vector>

#include "../../include/qre_moe.h"
#include "formats.cuh"
#include "internal.h"

// LRU state of one pool: a doubly linked list over the slots, least recent at
// the head; never-used slots start in index order (slot 0 least recent).
struct moe_slot_table {
  int nslots;
  std::vector<int> prev, next;
  int head, tail;
  std::vector<long long> key_of;                 // slot -> (layer, expert) key, -1 when never used
  std::unordered_map<long long, int> slot_of;    // key -> slot
  long long hits, misses;
};

struct moe_cache {
  moe_layer_geom geom;       // E = slots
  moe_slot_table* table;
  moe_bank* bank;            // the pool as a bank (borrows gu / dn)
  uint8_t* gu;               // [slots][2I][rb_gu] + slack
  uint8_t* dn;               // [slots][H][rb_dn] + slack
  size_t gu_expert, dn_expert;
  size_t gu_span, dn_span;   // bytes of each region, slack included
  bool owns_rows;            // false: carved from caller memory (moe_cache_create_at)
  long long h2d_bytes;
  std::vector<int32_t> fill_slots, fill_experts;
};

// One layer's whole bank at the start of an arena that pools also occupy
// (the full-layer prefill overlay): gate_up rows, then down rows.
struct moe_overlay {
  moe_layer_geom geom;
  uint8_t* base;
  size_t bytes;              // moe_overlay_bytes(geom)
  size_t gu_bytes, dn_bytes; // E * 2I * rb_gu, E * H * rb_dn
  moe_bank* bank;            // borrows [base, base + bytes)
};

namespace {

const float kOnes[4] = {1.0f, 1.0f, 1.0f, 1.0f};   // scale row of an expert whose layer has no scale bank

// One launch copies up to kFillMaxJobs contiguous byte ranges, cut into
// 16 KB chunks that the CTAs take in turn (kernel parameters stay < 4 KB).
constexpr int kFillMaxJobs = 120;
constexpr unsigned long long kFillChunk = 16384;
struct FillParams {
  int njobs;
  unsigned long long chunk0[kFillMaxJobs + 1];   // first chunk of each job; chunk0[njobs] = total
  const uint8_t* src[kFillMaxJobs];
  uint8_t* dst[kFillMaxJobs];
  unsigned long long bytes[kFillMaxJobs];
};

__global__ void __launch_bounds__(256) k_cache_fill(const __grid_constant__ FillParams p) {
  const unsigned long long total = p.chunk0[p.njobs];
  int j = 0;
  for (unsigned long long c = blockIdx.x; c < total; c += gridDim.x) {
    while (p.chunk0[j + 1] <= c) ++j;            // chunks are visited in increasing order
    const unsigned long long off = (c - p.chunk0[j]) * kFillChunk;
    const unsigned long long rest = p.bytes[j] - off;
    const unsigned long long n = rest < kFillChunk ? rest : kFillChunk;
    const uint8_t* s = p.src[j] + off;
    uint8_t* d = p.dst[j] + off;
    if (((reinterpret_cast<uintptr_t>(s) | reinterpret_cast<uintptr_t>(d) | n) & 15u) == 0) {
      const uint4* s4 = reinterpret_cast<const uint4*>(s);
      uint4* d4 = reinterpret_cast<uint4*>(d);
      for (unsigned long long i = threadIdx.x; i < n / 16; i += blockDim.x) d4[i] = s4[i];
    } else {
      for (unsigned long long i = threadIdx.x; i < n; i += blockDim.x) d[i] = s[i];
    }
  }
}

// The address the device uses for `p` when it may load from it directly
// (device or managed memory, or pinned host memory mapped into the device's
// address space), else nullptr.
const uint8_t* device_view(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged || a.type == cudaMemoryTypeHost)
    return static_cast<const uint8_t*>(a.devicePointer);
  return nullptr;
}

cudaError_t launch_fill(FillParams& fp, cudaStream_t s) {
  if (fp.njobs == 0) return cudaSuccess;
  const unsigned long long total = fp.chunk0[fp.njobs];
  const unsigned long long cap = 4ull * (unsigned long long)qre::sm_count();
  const int grid = (int)(total < cap ? total : cap);
  k_cache_fill<<<grid, 256, 0, s>>>(fp);
  fp.njobs = 0;
  fp.chunk0[0] = 0;
  return cudaGetLastError();
}

void add_fill(FillParams& fp, const uint8_t* src, uint8_t* dst, unsigned long long bytes) {
  const int j = fp.njobs++;
  fp.src[j] = src;
  fp.dst[j] = dst;
  fp.bytes[j] = bytes;
  fp.chunk0[j + 1] = fp.chunk0[j] + (bytes + kFillChunk - 1) / kFillChunk;
}

long long slot_key(int layer, int e) { return ((long long)(uint32_t)layer << 32) | (uint32_t)e; }

void lru_unlink(moe_slot_table* t, int s) {
  const int p = t->prev[s], n = t->next[s];
  if (p >= 0) t->next[p] = n; else t->head = n;
  if (n >= 0) t->prev[n] = p; else t->tail = p;
  t->prev[s] = t->next[s] = -1;
}

// Forget a slot's tag (its rows are not what the tag says): it stays where it
// is in the LRU order and holds no expert until filled again.
void slot_untag(moe_slot_table* t, int s) {
  if (t->key_of[s] >= 0) t->slot_of.erase(t->key_of[s]);
  t->key_of[s] = -1;
}

void lru_push_recent(moe_slot_table* t, int s) {
  t->prev[s] = t->tail;
  t->next[s] = -1;
  if (t->tail >= 0) t->next[t->tail] = s; else t->head = s;
  t->tail = s;
}

}  // namespace

int moe_slot_table_create(int32_t nslots, moe_slot_table** out) {
  if (!out || nslots < 1) return MOE_EINVAL;
  moe_slot_table* t = new (std::nothrow) moe_slot_table;
  if (!t) return MOE_ENOMEM;
  t->nslots = nslots;
  t->prev.assign(nslots, -1);
  t->next.assign(nslots, -1);
  t->key_of.assign(nslots, -1);
  t->head = t->tail = -1;
  for (int s = 0; s < nslots; ++s) lru_push_recent(t, s);
  t->hits = t->misses = 0;
  *out = t;
  return MOE_OK;
}

int moe_slot_table_destroy(moe_slot_table* t) {
  delete t;
  return MOE_OK;
}

int moe_slot_table_acquire(moe_slot_table* t, int32_t layer, const int32_t* ids, int32_t n, int32_t E,
                           int32_t* slot_ids, int32_t* fill_slots, int32_t* fill_experts, int32_t* nfill) {
  if (!t || (n > 0 && (!ids || !slot_ids)) || n < 0 || E < 1 || layer < 0 || !nfill) return MOE_EINVAL;
  // the request's distinct valid keys, in first-occurrence order
  std::vector<long long> keys;
  std::unordered_map<long long, int> seen;
  for (int i = 0; i < n; ++i) {
    const int e = ids[i];
    if (e < 0 || e >= E) continue;
    const long long k = slot_key(layer, e);
    if (seen.emplace(k, 1).second) keys.push_back(k);
  }
  if ((long long)keys.size() > t->nslots) return MOE_EUNSUPPORTED;
  if (!keys.empty() && (!fill_slots || !fill_experts)) return MOE_EINVAL;
  // hits become the most recent first, so no miss of this request evicts them
  for (const long long k : keys) {
    const auto it = t->slot_of.find(k);
    if (it == t->slot_of.end()) continue;
    lru_unlink(t, it->second);
    lru_push_recent(t, it->second);
    ++t->hits;
  }
  int nf = 0;
  for (const long long k : keys) {
    if (t->slot_of.count(k)) continue;
    const int s = t->head;   // least recent: neither a hit nor an earlier miss of this request
    lru_unlink(t, s);
    if (t->key_of[s] >= 0) t->slot_of.erase(t->key_of[s]);
    t->key_of[s] = k;
    t->slot_of[k] = s;
    lru_push_recent(t, s);
    ++t->misses;
    fill_slots[nf] = s;
    fill_experts[nf] = (int32_t)(k & 0xFFFFFFFFll);
    ++nf;
  }
  for (int i = 0; i < n; ++i) {
    const int e = ids[i];
    slot_ids[i] = (e < 0 || e >= E) ? -1 : t->slot_of[slot_key(layer, e)];
  }
  *nfill = nf;
  return MOE_OK;
}

int moe_slot_table_invalidate(moe_slot_table* t) {
  if (!t) return MOE_EINVAL;
  for (int s = 0; s < t->nslots; ++s) slot_untag(t, s);
  return MOE_OK;
}

int moe_slot_table_stats(const moe_slot_table* t, int64_t* hits, int64_t* misses) {
  if (!t) return MOE_EINVAL;
  if (hits) *hits = t->hits;
  if (misses) *misses = t->misses;
  return MOE_OK;
}

int moe_cache_plan(int64_t budget_bytes, int32_t ngeom, const int64_t* expert_bytes, const int64_t* selections,
                   int64_t* slots) {
  if (budget_bytes < 0 || ngeom < 1 || !expert_bytes || !selections || !slots) return MOE_EINVAL;
  __int128 unit = 0;
  for (int g = 0; g < ngeom; ++g) {
    if (expert_bytes[g] < 1 || selections[g] < 0) return MOE_EINVAL;
    unit += (__int128)selections[g] * expert_bytes[g];
  }
  __int128 left = budget_bytes;
  for (int g = 0; g < ngeom; ++g) {
    slots[g] = unit > 0 ? (int64_t)((__int128)budget_bytes * selections[g] / unit) : 0;
    left -= (__int128)slots[g] * expert_bytes[g];
  }
  // the bytes left over: one slot at a time of the smallest size that fits
  for (;;) {
    int best = -1;
    for (int g = 0; g < ngeom; ++g)
      if (expert_bytes[g] <= left && (best < 0 || expert_bytes[g] < expert_bytes[best])) best = g;
    if (best < 0) break;
    ++slots[best];
    left -= expert_bytes[best];
  }
  return MOE_OK;
}

namespace {

size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

// Bytes of a pool's rows: the gate_up region then the down region, each with
// 256 bytes of slack (a tensor-map tile of the last slot reads a whole box).
bool pool_spans(const moe_layer_geom& g, int32_t nslots, size_t& gu_expert, size_t& dn_expert, size_t& gu_span,
                size_t& dn_span) {
  const int rb_gu = qre::row_bytes_of(g.gate_up_type, g.H), rb_dn = qre::row_bytes_of(g.down_type, g.I);
  if (rb_gu == 0 || rb_dn == 0) return false;
  gu_expert = (size_t)2 * g.I * rb_gu;
  dn_expert = (size_t)g.H * rb_dn;
  gu_span = align256(gu_expert * nslots + 256);
  dn_span = align256(dn_expert * nslots + 256);
  return true;
}

// The pool over rows at gu / dn (owned or carved), zeroed on `stream`.
int cache_make(const moe_layer_geom* geom, int32_t nslots, uint8_t* gu, uint8_t* dn, bool owns, void* stream,
               moe_cache** out) {
  moe_layer_geom g = *geom;
  g.E = nslots;
  moe_cache* c = new (std::nothrow) moe_cache;
  if (!c) return MOE_ENOMEM;
  c->geom = g;
  pool_spans(g, nslots, c->gu_expert, c->dn_expert, c->gu_span, c->dn_span);
  c->h2d_bytes = 0;
  c->gu = gu;
  c->dn = dn;
  c->owns_rows = owns;
  c->bank = nullptr;
  c->table = nullptr;
  int st = moe_slot_table_create(nslots, &c->table);
  if (st) { delete c; return st; }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // defined contents for slots that were never filled (a decode may only
  // route to filled slots, but the tensor-map tiles of a slot read a whole box)
  cudaError_t e = cudaMemsetAsync(c->gu, 0, c->gu_span, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(c->dn, 0, c->dn_span, s);
  if (e == cudaSuccess)
    st = moe_bank_create(&g, c->gu, c->gu_expert * nslots, c->dn, c->dn_expert * nslots, nullptr,
                         MOE_SRC_DEVICE_BORROW, stream, &c->bank);
  if (e != cudaSuccess || st != MOE_OK) {
    moe_slot_table_destroy(c->table);
    delete c;
    return e != cudaSuccess ? qre::report_cuda_error(e, "cache create") : st;
  }
  c->fill_slots.resize(nslots);
  c->fill_experts.resize(nslots);
  *out = c;
  return MOE_OK;
}

}  // namespace

int moe_cache_create(const moe_layer_geom* geom, int32_t nslots, void* stream, moe_cache** out) {
  if (!geom || !out || nslots < 1 || nslots > MOE_MAX_E) return MOE_EINVAL;
  size_t ge, de, gs, ds;
  if (!pool_spans(*geom, nslots, ge, de, gs, ds)) return MOE_EINVAL;
  uint8_t *gu = nullptr, *dn = nullptr;
  if (cudaMalloc(&gu, gs) != cudaSuccess || cudaMalloc(&dn, ds) != cudaSuccess) {
    cudaGetLastError();
    cudaFree(gu); cudaFree(dn);
    return MOE_ENOMEM;
  }
  const int st = cache_make(geom, nslots, gu, dn, true, stream, out);
  if (st) { cudaFree(gu); cudaFree(dn); }
  return st;
}

size_t moe_cache_bytes(const moe_layer_geom* geom, int32_t nslots) {
  if (!geom || nslots < 1 || nslots > MOE_MAX_E) return 0;
  size_t ge, de, gs, ds;
  if (!pool_spans(*geom, nslots, ge, de, gs, ds)) return 0;
  return gs + ds;
}

int moe_cache_create_at(const moe_layer_geom* geom, int32_t nslots, void* base, size_t bytes, void* stream,
                        moe_cache** out) {
  if (!geom || !out || !base || nslots < 1 || nslots > MOE_MAX_E) return MOE_EINVAL;
  if ((reinterpret_cast<uintptr_t>(base) & 255) != 0) return MOE_EINVAL;
  const size_t need = moe_cache_bytes(geom, nslots);
  if (need == 0 || bytes < need) return MOE_EINVAL;
  size_t ge = 0, de = 0, gs = 0, ds = 0;
  if (!pool_spans(*geom, nslots, ge, de, gs, ds)) return MOE_EINVAL;
  uint8_t* gu = static_cast<uint8_t*>(base);
  return cache_make(geom, nslots, gu, gu + gs, false, stream, out);
}

int moe_cache_invalidate(moe_cache* c) {
  if (!c) return MOE_EINVAL;
  return moe_slot_table_invalidate(c->table);
}

int moe_cache_destroy(moe_cache* c) {
  if (!c) return MOE_OK;
  moe_bank_destroy(c->bank);   // synchronizes the device
  if (c->owns_rows) {
    cudaFree(c->gu);
    cudaFree(c->dn);
  }
  moe_slot_table_destroy(c->table);
  delete c;
  return MOE_OK;
}

moe_bank* moe_cache_bank(moe_cache* c) { return c ? c->bank : nullptr; }

int moe_cache_acquire(moe_cache* c, int32_t layer, const void* gate_up, const void* down, const float* scales,
                      int32_t E, const int32_t* ids, int32_t n, int32_t* slot_ids, int32_t* nfill, void* stream) {
  if (!c || !gate_up || !down || E < 1) return MOE_EINVAL;
  int32_t nf = 0;
  const int st = moe_slot_table_acquire(c->table, layer, ids, n, E, slot_ids, c->fill_slots.data(),
                                        c->fill_experts.data(), &nf);
  if (st) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  float* sdev = qre::bank_scales(c->bank);
  const uint8_t* gsrc = static_cast<const uint8_t*>(gate_up);
  const uint8_t* dsrc = static_cast<const uint8_t*>(down);
  // rows the device can load directly are copied by one kernel per request
  const uint8_t* gview = nf > 0 ? device_view(gate_up) : nullptr;
  const uint8_t* dview = nf > 0 ? device_view(down) : nullptr;
  const bool by_kernel = gview && dview;
  FillParams fp;
  fp.njobs = 0;
  fp.chunk0[0] = 0;
  for (int i = 0; i < nf; ++i) {
    const size_t slot = (size_t)c->fill_slots[i], e = (size_t)c->fill_experts[i];
    cudaError_t err = cudaSuccess;
    if (by_kernel) {
      if (fp.njobs + 2 > kFillMaxJobs) err = launch_fill(fp, s);
      add_fill(fp, gview + e * c->gu_expert, c->gu + slot * c->gu_expert, c->gu_expert);
      add_fill(fp, dview + e * c->dn_expert, c->dn + slot * c->dn_expert, c->dn_expert);
    } else {
      err = cudaMemcpyAsync(c->gu + slot * c->gu_expert, gsrc + e * c->gu_expert, c->gu_expert, cudaMemcpyDefault,
                            s);
      if (err == cudaSuccess)
        err = cudaMemcpyAsync(c->dn + slot * c->dn_expert, dsrc + e * c->dn_expert, c->dn_expert,
                              cudaMemcpyDefault, s);
    }
    if (err == cudaSuccess)
      err = cudaMemcpyAsync(sdev + 4 * slot, scales ? scales + 4 * e : kOnes, 16, cudaMemcpyDefault, s);
    if (err != cudaSuccess) {
      for (int k = 0; k < nf; ++k) slot_untag(c->table, c->fill_slots[k]);   // none of this request's fills counts
      return qre::report_cuda_error(err, "cache fill");
    }
    c->h2d_bytes += (long long)(c->gu_expert + c->dn_expert + 16);
  }
  if (by_kernel) {
    const cudaError_t err = launch_fill(fp, s);
    if (err != cudaSuccess) {
      for (int k = 0; k < nf; ++k) slot_untag(c->table, c->fill_slots[k]);
      return qre::report_cuda_error(err, "cache fill");
    }
  }
  if (nfill) *nfill = nf;
  return MOE_OK;
}

int moe_cache_stats(const moe_cache* c, int64_t* hits, int64_t* misses, int64_t* copied_bytes) {
  if (!c) return MOE_EINVAL;
  moe_slot_table_stats(c->table, hits, misses);
  if (copied_bytes) *copied_bytes = c->h2d_bytes;
  return MOE_OK;
}

// ------------------------------------------------------------------ full-layer prefill overlay

size_t moe_overlay_bytes(const moe_layer_geom* geom) {
  if (!geom || geom->E < 1 || geom->E > MOE_MAX_E) return 0;
  const int rb_gu = qre::row_bytes_of(geom->gate_up_type, geom->H), rb_dn = qre::row_bytes_of(geom->down_type, geom->I);
  if (rb_gu == 0 || rb_dn == 0) return 0;
  return align256((size_t)geom->E * 2 * geom->I * rb_gu + 256) + align256((size_t)geom->E * geom->H * rb_dn + 256);
}

int moe_overlay_create(const moe_layer_geom* geom, void* base, size_t bytes, void* stream, moe_overlay** out) {
  if (!geom || !base || !out) return MOE_EINVAL;
  if ((reinterpret_cast<uintptr_t>(base) & 255) != 0) return MOE_EINVAL;
  const size_t need = moe_overlay_bytes(geom);
  if (need == 0 || bytes < need) return MOE_EINVAL;
  moe_overlay* ov = new (std::nothrow) moe_overlay;
  if (!ov) return MOE_ENOMEM;
  ov->geom = *geom;
  ov->base = static_cast<uint8_t*>(base);
  ov->bytes = need;
  ov->gu_bytes = (size_t)geom->E * 2 * geom->I * qre::row_bytes_of(geom->gate_up_type, geom->H);
  ov->dn_bytes = (size_t)geom->E * geom->H * qre::row_bytes_of(geom->down_type, geom->I);
  ov->bank = nullptr;
  const int st = moe_bank_create(geom, ov->base, ov->gu_bytes, ov->base + align256(ov->gu_bytes + 256), ov->dn_bytes,
                                 nullptr, MOE_SRC_DEVICE_BORROW, stream, &ov->bank);
  if (st) {
    delete ov;
    return st;
  }
  *out = ov;
  return MOE_OK;
}

int moe_overlay_destroy(moe_overlay* ov) {
  if (!ov) return MOE_OK;
  moe_bank_destroy(ov->bank);
  delete ov;
  return MOE_OK;
}

moe_bank* moe_overlay_bank(moe_overlay* ov) { return ov ? ov->bank : nullptr; }

int moe_overlay_load(moe_overlay* ov, moe_cache* const* pools, int32_t npools, const void* gate_up, const void* down,
                     const float* scales, void* stream) {
  if (!ov || !gate_up || !down || npools < 0 || (npools > 0 && !pools)) return MOE_EINVAL;
  // every pool whose rows share bytes with the overlay loses its tags before
  // anything is copied (the pages' order: invalidate, then write the overlay)
  const uintptr_t o0 = reinterpret_cast<uintptr_t>(ov->base), o1 = o0 + ov->bytes;
  for (int i = 0; i < npools; ++i) {
    moe_cache* c = pools[i];
    if (!c) return MOE_EINVAL;
    const uintptr_t g0 = reinterpret_cast<uintptr_t>(c->gu), g1 = g0 + c->gu_span;
    const uintptr_t d0 = reinterpret_cast<uintptr_t>(c->dn), d1 = d0 + c->dn_span;
    if ((g0 < o1 && o0 < g1) || (d0 < o1 && o0 < d1)) moe_slot_table_invalidate(c->table);
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* gdst = ov->base;
  uint8_t* ddst = ov->base + align256(ov->gu_bytes + 256);
  const uint8_t* gview = device_view(gate_up);
  const uint8_t* dview = device_view(down);
  cudaError_t e;
  if (gview && dview) {
    FillParams fp;
    fp.njobs = 0;
    fp.chunk0[0] = 0;
    add_fill(fp, gview, gdst, ov->gu_bytes);
    add_fill(fp, dview, ddst, ov->dn_bytes);
    e = launch_fill(fp, s);
  } else {
    e = cudaMemcpyAsync(gdst, gate_up, ov->gu_bytes, cudaMemcpyDefault, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(ddst, down, ov->dn_bytes, cudaMemcpyDefault, s);
  }
  float* sdev = qre::bank_scales(ov->bank);
  for (int ex = 0; e == cudaSuccess && ex < (scales ? 1 : ov->geom.E); ++ex)
    e = scales ? cudaMemcpyAsync(sdev, scales, 16 * (size_t)ov->geom.E, cudaMemcpyDefault, s)
               : cudaMemcpyAsync(sdev + 4 * ex, kOnes, 16, cudaMemcpyHostToDevice, s);
  return e == cudaSuccess ? MOE_OK : qre::report_cuda_error(e, "overlay load");
}
