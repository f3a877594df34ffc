// Unified page pool: host bookkeeping, device page tables, adapter loading, status.
//
// "S-LoRA, in depth", section "Unified paging: adapters and KV cache in one pool":
// one page holds one H-vector; KV cache and adapters draw pages from one free list;
// a rank-r A or B takes r pages.  The pool sketch there pops its free list from the
// end and appends freed pages; this pool keeps that order so that page placement is
// reproducible from the initial free-list order.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdio>
#include <cstring>
#include <new>
#include <string>
#include <thread>

#include "lora_internal.h"

namespace {
thread_local std::string g_last_error;

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// The columns of A (H x rank, row-major) as rank page rows of H values.  Blocked over 64 rows
// of A at a time: the block's reads stay in the first-level cache and every row receives 64
// contiguous values per block (a column-by-column walk strides through all of A per column).
void columns_to_rows(const uint16_t* A, int64_t H, int rank, uint16_t* rows) {
  constexpr int64_t kBlock = 64;
  for (int64_t k0 = 0; k0 < H; k0 += kBlock) {
    const int64_t k1 = std::min(H, k0 + kBlock);
    for (int j = 0; j < rank; ++j) {
      uint16_t* dst = rows + (int64_t)j * H;
      for (int64_t k = k0; k < k1; ++k) dst[k] = A[k * rank + j];
    }
  }
}

// An adapter's page rows, slot after slot (A's columns, then B's rows), into `rows`.  Slots are
// independent, so a large adapter is split over up to 8 host threads (a host at one thread's
// copy rate repacks a 32 MiB adapter in several ms); if a thread cannot be started, the calling
// thread does its share.
void pack_rows(const void* const* A_host, const void* const* B_host, const std::vector<uint8_t>& present, int64_t H,
               int rank, uint16_t* rows) {
  std::vector<int> slots;
  for (int s = 0; s < (int)present.size(); ++s)
    if (present[s]) slots.push_back(s);
  const size_t n = slots.size();
  auto one = [&](size_t i) {
    const int s = slots[i];
    uint16_t* out = rows + (int64_t)i * 2 * rank * H;
    columns_to_rows(static_cast<const uint16_t*>(A_host[s]), H, rank, out);
    std::memcpy(out + (int64_t)rank * H, B_host[s], (size_t)rank * H * sizeof(uint16_t));
  };
  unsigned nt = std::min(std::max(1u, std::thread::hardware_concurrency()), 8u);
  if (n * 2 * rank * H * sizeof(uint16_t) < (8u << 20)) nt = 1;
  nt = (unsigned)std::min<size_t>(nt, std::max<size_t>(n, 1));
  auto share = [&](unsigned t) {
    for (size_t i = t; i < n; i += nt) one(i);
  };
  std::vector<std::thread> threads;
  unsigned started = 1;                          // share 0 is the calling thread's
  try {
    for (; started < nt; ++started) threads.emplace_back(share, started);
  } catch (...) {
  }
  for (unsigned t = started; t < nt; ++t) share(t);
  share(0);
  for (auto& th : threads) th.join();
}

// Copy staged rows (page ids first, then the rows in the same order) into their pages.
__global__ void scatter_pages_kernel(const int32_t* __restrict__ ids, const uint4* __restrict__ rows,
                                     int64_t n_pages, int32_t H, uint4* __restrict__ pool) {
  const int64_t vec_per_row = H / 8;   // 8 bf16 per 16-byte vector
  for (int64_t r = blockIdx.x; r < n_pages; r += gridDim.x) {
    const int64_t page = ids[r];
    const uint4* src = rows + r * vec_per_row;
    uint4* dst = pool + page * vec_per_row;
    for (int64_t v = threadIdx.x; v < vec_per_row; v += blockDim.x) dst[v] = src[v];
  }
}

// Copy packed page rows, read straight from pinned host memory, into their pages; block 0 also
// writes the adapter's device page table and rank.  Users of the adapter wait for the kernel
// (an event on its stream) before reading either.
__global__ void load_packed_kernel(const int32_t* __restrict__ ids, const int32_t* __restrict__ tab_image,
                                   const uint4* __restrict__ rows, int64_t n_pages, int32_t H,
                                   uint4* __restrict__ pool, int32_t* __restrict__ d_tab, int32_t n_tab,
                                   int32_t* __restrict__ d_rank, int32_t rank) {
  const int64_t vec_per_row = H / 8;
  for (int64_t r = blockIdx.x; r < n_pages; r += gridDim.x) {
    const int64_t page = ids[r];
    const uint4* src = rows + r * vec_per_row;
    uint4* dst = pool + page * vec_per_row;
    for (int64_t v = threadIdx.x; v < vec_per_row; v += blockDim.x) dst[v] = src[v];
  }
  if (blockIdx.x == 0) {
    for (int i = threadIdx.x; i < n_tab; i += blockDim.x) d_tab[i] = tab_image[i];
    if (threadIdx.x == 0) *d_rank = rank;
  }
}

// Byte layout of a packed adapter: page ids [need] int32, the device page-table image
// [n_slots][2][64] int32, then the page rows [need][H] bf16; each part 256-byte aligned.
struct PackedLayout {
  int64_t need;
  size_t ids, tab, rows, total;
};
PackedLayout packed_layout(const lora_pool* p, int32_t rank, int64_t n_present) {
  PackedLayout L;
  L.need = 2 * (int64_t)rank * n_present;
  L.ids = 0;
  L.tab = align_up((size_t)L.need * sizeof(int32_t), 256);
  L.rows = L.tab + align_up((size_t)p->n_slots * kTabStride * sizeof(int32_t), 256);
  L.total = L.rows + (size_t)L.need * p->H * sizeof(uint16_t);
  return L;
}
}  // namespace

int device_sm_count() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        n <= 0)
      n = 148;
  }
  return n;
}

int lora_fail(int code, const std::string& msg) {
  g_last_error = msg;
  return code;
}

int lora_cuda_fail(cudaError_t e, const char* what) {
  return lora_fail(LORA_ECUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

int launch_scatter_pages(const uint16_t* stage, const int32_t* d_pages, int64_t n_pages, int32_t H,
                         void* pool_dev, cudaStream_t st) {
  (void)stage;
  if (n_pages == 0) return LORA_OK;
  const size_t ids_bytes = align_up(n_pages * sizeof(int32_t), 256);
  const uint4* rows = reinterpret_cast<const uint4*>(reinterpret_cast<const char*>(d_pages) + ids_bytes);
  int grid = (int)std::min<int64_t>(n_pages, 4096);
  scatter_pages_kernel<<<grid, 256, 0, st>>>(d_pages, rows, n_pages, H, reinterpret_cast<uint4*>(pool_dev));
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? LORA_OK : lora_cuda_fail(e, "scatter_pages launch");
}

namespace {
cudaEvent_t take_event(lora_pool* p) {
  if (!p->ev_free.empty()) {
    cudaEvent_t e = p->ev_free.back();
    p->ev_free.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}
}  // namespace

ProfScope::ProfScope(const lora_pool* pool, int k, cudaStream_t s) : p(const_cast<lora_pool*>(pool)), kind(k), st(s) {
  if (!p) return;                       // a launch made for no pool (nothing to count)
  p->launches[kind] += 1;
  if (!p->prof_on) return;
  cudaEvent_t a = take_event(p), b = take_event(p);
  if (!a || !b) return;
  // While the stream is being captured into a graph, records must be external to become event
  // nodes of the graph; on an ordinary stream a plain record is the valid form.
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  (void)cudaStreamIsCapturing(st, &cs);
  capturing = cs == cudaStreamCaptureStatusActive;
  const cudaError_t e = capturing ? cudaEventRecordWithFlags(a, st, cudaEventRecordExternal) : cudaEventRecord(a, st);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();           // profiling must not turn into a launch error
    return;
  }
  p->prof_rec.push_back({kind, a, b});
  rec = (int)p->prof_rec.size() - 1;
}

ProfScope::~ProfScope() {
  if (rec < 0) return;
  const cudaEvent_t b = p->prof_rec[rec].stop;
  const cudaError_t e = capturing ? cudaEventRecordWithFlags(b, st, cudaEventRecordExternal) : cudaEventRecord(b, st);
  if (e != cudaSuccess) (void)cudaGetLastError();
}

extern "C" {

const char* lora_last_error(void) { return g_last_error.c_str(); }

int lora_profile_enable(lora_pool* p, int32_t enable) {
  if (!p) return lora_fail(LORA_EINVAL, "lora_profile_enable: pool is NULL");
  if (p->planning && enable) return lora_fail(LORA_EINVAL, "lora_profile_enable: planning pool launches nothing");
  p->prof_on = enable != 0;
  return LORA_OK;
}

int lora_profile_read(lora_pool* p, int32_t n_kinds, int64_t* launches, double* ms, int32_t reset) {
  if (!p || n_kinds < 0 || (n_kinds > 0 && (!launches || !ms))) return lora_fail(LORA_EINVAL, "lora_profile_read: bad arguments");
  double acc[LORA_N_KINDS] = {};
  int rc = LORA_OK;
  for (auto& r : p->prof_rec) {
    float t = 0.f;
    cudaError_t e = cudaEventSynchronize(r.stop);
    if (e == cudaSuccess) e = cudaEventElapsedTime(&t, r.start, r.stop);
    if (e == cudaErrorInvalidResourceHandle) {   // captured into a graph that has not run yet
      (void)cudaGetLastError();                  // do not leave it as the runtime's last error
      e = cudaSuccess;
      t = 0.f;
    }
    if (e != cudaSuccess && rc == LORA_OK) rc = lora_cuda_fail(e, "lora_profile_read");
    acc[r.kind] += t;
  }
  for (int k = 0; k < n_kinds; ++k) {
    launches[k] = k < LORA_N_KINDS ? p->launches[k] : 0;
    ms[k] = k < LORA_N_KINDS ? acc[k] : 0.0;
  }
  if (reset) {
    for (auto& r : p->prof_rec) {
      p->ev_free.push_back(r.start);
      p->ev_free.push_back(r.stop);
    }
    p->prof_rec.clear();
    for (int k = 0; k < LORA_N_KINDS; ++k) p->launches[k] = 0;
  }
  return rc;
}

int lora_pool_create(void* pool_dev, int64_t num_pages, int32_t H, int32_t n_slots, int32_t max_adapters,
                     const int64_t* page_order_host, lora_pool** out) {
  if (!out) return lora_fail(LORA_EINVAL, "lora_pool_create: out is NULL");
  *out = nullptr;
  if (num_pages < 1 || num_pages > INT32_MAX)
    return lora_fail(LORA_EINVAL, "lora_pool_create: num_pages must be in [1, 2^31-1]");
  if (H < 64 || H > 16384 || H % 64 != 0)
    return lora_fail(LORA_EINVAL, "lora_pool_create: H must be a multiple of 64 in [64, 16384]");
  if (n_slots < 1) return lora_fail(LORA_EINVAL, "lora_pool_create: n_slots must be >= 1");
  if (max_adapters < 1 || max_adapters > LORA_MAX_ADAPTERS)
    return lora_fail(LORA_EINVAL, "lora_pool_create: max_adapters must be in [1, LORA_MAX_ADAPTERS]");
  if ((reinterpret_cast<uintptr_t>(pool_dev) & 15) != 0)
    return lora_fail(LORA_EINVAL, "lora_pool_create: pool storage must be 16-byte aligned");

  lora_pool* p = new (std::nothrow) lora_pool();
  if (!p) return lora_fail(LORA_EINVAL, "lora_pool_create: out of host memory");
  p->pool_dev = pool_dev;
  p->num_pages = num_pages;
  p->H = H;
  p->n_slots = n_slots;
  p->max_adapters = max_adapters;
  p->planning = (pool_dev == nullptr);
  p->page_state.assign(num_pages, 0);
  p->free_list.resize(num_pages);
  if (page_order_host) {
    std::vector<uint8_t> seen(num_pages, 0);
    for (int64_t i = 0; i < num_pages; ++i) {
      const int64_t v = page_order_host[i];
      if (v < 0 || v >= num_pages || seen[v]) {
        delete p;
        return lora_fail(LORA_EINVAL, "lora_pool_create: page_order is not a permutation of 0..num_pages-1");
      }
      seen[v] = 1;
      p->free_list[i] = (int32_t)v;
    }
  } else {
    for (int64_t i = 0; i < num_pages; ++i) p->free_list[i] = (int32_t)i;
  }
  p->rank.assign(max_adapters, 0);
  p->tables.resize(max_adapters);
  p->refs.assign(max_adapters, 0);
  p->load_seq.assign(max_adapters, 0);
  p->last_use.assign(max_adapters, 0);
  p->ev_ready.assign(max_adapters, nullptr);
  p->ready_pending.assign(max_adapters, 0);

  if (!p->planning) {
    cudaError_t e = cudaGetDevice(&p->device);
    const size_t tab_bytes = (size_t)max_adapters * n_slots * kTabStride * sizeof(int32_t);
    if (e == cudaSuccess) e = cudaMalloc(&p->d_ptab, tab_bytes);
    if (e == cudaSuccess) e = cudaMalloc(&p->d_rank, (size_t)max_adapters * sizeof(int32_t));
    if (e == cudaSuccess) e = cudaMalloc(&p->d_err, 4 * sizeof(int32_t));
    if (e == cudaSuccess) e = cudaMemset(p->d_ptab, 0xFF, tab_bytes);
    if (e == cudaSuccess) e = cudaMemset(p->d_rank, 0, (size_t)max_adapters * sizeof(int32_t));
    if (e == cudaSuccess) e = cudaMemset(p->d_err, 0, 4 * sizeof(int32_t));
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
      lora_pool_destroy(p);
      return lora_cuda_fail(e, "lora_pool_create");
    }
  }
  *out = p;
  return LORA_OK;
}

void lora_pool_destroy(lora_pool* p) {
  if (!p) return;
  for (auto& r : p->prof_rec) {
    cudaEventDestroy(r.start);
    cudaEventDestroy(r.stop);
  }
  for (auto e : p->ev_free) cudaEventDestroy(e);
  for (auto e : p->ev_ready)
    if (e) cudaEventDestroy(e);
  if (p->ev_freed) cudaEventDestroy(p->ev_freed);
  if (p->d_ptab) cudaFree(p->d_ptab);
  if (p->d_rank) cudaFree(p->d_rank);
  if (p->d_err) cudaFree(p->d_err);
  if (p->d_stage) cudaFree(p->d_stage);
  delete p;
}

int lora_pool_reserve(lora_pool* p, int64_t n, int64_t* ids) {
  if (!p || n < 0 || (n > 0 && !ids)) return lora_fail(LORA_EINVAL, "lora_pool_reserve: bad arguments");
  if (n > (int64_t)p->free_list.size())
    return lora_fail(LORA_ENOPAGES, "lora_pool_reserve: " + std::to_string(n) + " pages asked, " +
                                        std::to_string(p->free_list.size()) + " free");
  for (int64_t i = 0; i < n; ++i) {
    const int32_t pg = p->free_list.back();
    p->free_list.pop_back();
    p->page_state[pg] = 1;
    ids[i] = pg;
  }
  p->reserved_pages += n;
  return LORA_OK;
}

int lora_kv_grow(lora_pool* p, int64_t request, int32_t n_tokens, int32_t layers, int32_t* ids_out) {
  if (!p || n_tokens < 0 || layers < 1) return lora_fail(LORA_EINVAL, "lora_kv_grow: bad arguments");
  auto it = p->kv.find(request);
  if (it != p->kv.end() && it->second.layers != layers)
    return lora_fail(LORA_EINVAL, "lora_kv_grow: request " + std::to_string(request) + " has " +
                                      std::to_string(it->second.layers) + " layers");
  const int64_t need = 2 * (int64_t)layers * n_tokens;
  if (need > (int64_t)p->free_list.size())
    return lora_fail(LORA_ENOPAGES, "lora_kv_grow: " + std::to_string(need) + " pages asked, " +
                                        std::to_string(p->free_list.size()) + " free");
  auto& req = p->kv[request];
  req.layers = layers;
  for (int64_t i = 0; i < need; ++i) {
    const int32_t pg = p->free_list.back();
    p->free_list.pop_back();
    p->page_state[pg] = 4;
    req.pages.push_back(pg);
    if (ids_out) ids_out[i] = pg;
  }
  p->reserved_pages += need;
  return LORA_OK;
}

int lora_kv_free(lora_pool* p, int64_t request) {
  if (!p) return lora_fail(LORA_EINVAL, "lora_kv_free: pool is NULL");
  auto it = p->kv.find(request);
  if (it == p->kv.end()) return lora_fail(LORA_EINVAL, "lora_kv_free: request " + std::to_string(request) + " holds no pages");
  for (int32_t pg : it->second.pages) {
    p->page_state[pg] = 0;
    p->free_list.push_back(pg);
  }
  p->reserved_pages -= (int64_t)it->second.pages.size();
  p->kv.erase(it);
  return LORA_OK;
}

int64_t lora_kv_length(const lora_pool* p, int64_t request) {
  if (!p) return -1;
  auto it = p->kv.find(request);
  if (it == p->kv.end()) return -1;
  return (int64_t)it->second.pages.size() / (2 * it->second.layers);
}

int lora_kv_table(const lora_pool* p, int64_t request, int32_t layer, int32_t* table) {
  if (!p || !table) return lora_fail(LORA_EINVAL, "lora_kv_table: bad arguments");
  auto it = p->kv.find(request);
  if (it == p->kv.end()) return lora_fail(LORA_EINVAL, "lora_kv_table: request " + std::to_string(request) + " holds no pages");
  const int32_t L = it->second.layers;
  if (layer < 0 || layer >= L) return lora_fail(LORA_EINVAL, "lora_kv_table: layer out of range");
  const int64_t n = (int64_t)it->second.pages.size() / (2 * L);
  for (int64_t t = 0; t < n; ++t) {
    table[2 * t] = it->second.pages[(t * L + layer) * 2];
    table[2 * t + 1] = it->second.pages[(t * L + layer) * 2 + 1];
  }
  return LORA_OK;
}

int lora_pool_release(lora_pool* p, int64_t n, const int64_t* ids) {
  if (!p || n < 0 || (n > 0 && !ids)) return lora_fail(LORA_EINVAL, "lora_pool_release: bad arguments");
  int64_t i = 0;
  for (; i < n; ++i) {   // validate, marking as we go so duplicates are caught
    const int64_t pg = ids[i];
    if (pg < 0 || pg >= p->num_pages || p->page_state[pg] != 1) break;
    p->page_state[pg] = 3;
  }
  if (i < n) {
    for (int64_t k = 0; k < i; ++k) p->page_state[ids[k]] = 1;
    return lora_fail(LORA_EINVAL, "lora_pool_release: page " + std::to_string(ids[i]) +
                                      " is not reserved or is listed twice");
  }
  for (int64_t k = 0; k < n; ++k) {
    p->page_state[ids[k]] = 0;
    p->free_list.push_back((int32_t)ids[k]);
  }
  p->reserved_pages -= n;
  return LORA_OK;
}

int lora_adapter_load(lora_pool* p, int32_t aid, int32_t rank, const void* const* A_host,
                      const void* const* B_host, lora_stream_t stream, int32_t* table_out) {
  if (!p) return lora_fail(LORA_EINVAL, "lora_adapter_load: pool is NULL");
  if (aid < 0 || aid >= p->max_adapters)
    return lora_fail(LORA_EINVAL, "lora_adapter_load: adapter id " + std::to_string(aid) + " outside [0, max_adapters)");
  if (rank < 1 || rank > LORA_MAX_RANK)
    return lora_fail(LORA_ERANK, "lora_adapter_load: rank " + std::to_string(rank) + " outside [1, 64]");
  if (p->rank[aid] != 0) return lora_fail(LORA_EEXIST, "lora_adapter_load: adapter " + std::to_string(aid) + " already loaded");
  if (!p->planning && (!A_host || !B_host))
    return lora_fail(LORA_EINVAL, "lora_adapter_load: A_host and B_host arrays are required");
  const int S = p->n_slots;
  std::vector<uint8_t> present(S, 1);
  if (A_host)
    for (int s = 0; s < S; ++s) present[s] = A_host[s] != nullptr;
  if (!p->planning)
    for (int s = 0; s < S; ++s)
      if (present[s] && !B_host[s]) return lora_fail(LORA_EINVAL, "lora_adapter_load: B_host[slot] is NULL where A_host[slot] is set");
  int64_t n_present = 0;
  for (int s = 0; s < S; ++s) n_present += present[s];
  const int64_t need = 2 * (int64_t)rank * n_present;
  if (need > (int64_t)p->free_list.size())
    return lora_fail(LORA_ENOPAGES, "lora_adapter_load: adapter needs " + std::to_string(need) + " pages, " +
                                        std::to_string(p->free_list.size()) + " free");

  // Take pages: slot-major, A then B, j ascending, each from the end of the free list.
  std::vector<int32_t> table((size_t)S * 2 * rank, -1);
  std::vector<int32_t> taken;
  taken.reserve(need);
  for (int s = 0; s < S; ++s) {
    if (!present[s]) continue;
    for (int half = 0; half < 2; ++half)
      for (int j = 0; j < rank; ++j) {
        const int32_t pg = p->free_list.back();
        p->free_list.pop_back();
        table[((size_t)s * 2 + half) * rank + j] = pg;
        taken.push_back(pg);
      }
  }
  auto rollback = [&]() {
    for (auto it = taken.rbegin(); it != taken.rend(); ++it) p->free_list.push_back(*it);
  };

  if (!p->planning) {
    const int64_t H = p->H;
    const size_t ids_bytes = align_up(need * sizeof(int32_t), 256);
    const size_t bytes = ids_bytes + (size_t)need * H * sizeof(uint16_t);
    p->h_stage.resize((bytes + 1) / 2);
    char* base = reinterpret_cast<char*>(p->h_stage.data());
    std::memcpy(base, taken.data(), need * sizeof(int32_t));
    uint16_t* rows = reinterpret_cast<uint16_t*>(base + ids_bytes);
    pack_rows(A_host, B_host, present, H, rank, rows);
    cudaError_t e = cudaSuccess;
    if (bytes > p->d_stage_bytes) {
      if (p->d_stage) cudaFree(p->d_stage);
      p->d_stage = nullptr;
      p->d_stage_bytes = 0;
      e = cudaMalloc(&p->d_stage, bytes);
      if (e == cudaSuccess) p->d_stage_bytes = bytes;
    }
    std::vector<int32_t> dtab((size_t)S * kTabStride, -1);
    for (int s = 0; s < S; ++s)
      for (int half = 0; half < 2; ++half)
        for (int j = 0; j < rank; ++j) dtab[(size_t)s * kTabStride + half * LORA_MAX_RANK + j] = table[((size_t)s * 2 + half) * rank + j];
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (e == cudaSuccess && p->freed_recorded) e = cudaStreamWaitEvent(st, p->ev_freed, 0);   // pages reused
    if (e == cudaSuccess) e = cudaMemcpyAsync(p->d_stage, base, bytes, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) {
      ProfScope prof(p, LORA_KIND_SCATTER, st);
      int rc = launch_scatter_pages(nullptr, static_cast<const int32_t*>(p->d_stage), need, p->H, p->pool_dev, st);
      if (rc != LORA_OK) e = cudaErrorLaunchFailure;
    }
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(p->d_ptab + (size_t)aid * S * kTabStride, dtab.data(), dtab.size() * sizeof(int32_t),
                          cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(p->d_rank + aid, &rank, sizeof(int32_t), cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) {
      rollback();
      return lora_cuda_fail(e, "lora_adapter_load");
    }
  }
  for (int32_t pg : taken) p->page_state[pg] = 2;
  p->rank[aid] = rank;
  p->refs[aid] = 0;
  p->load_seq[aid] = p->next_seq++;
  p->last_use[aid] = ++p->use_clock;
  p->tables[aid] = table;
  p->adapter_pages += need;
  p->resident += 1;
  if (table_out) std::memcpy(table_out, table.data(), table.size() * sizeof(int32_t));
  return LORA_OK;
}

}  // extern "C"

namespace {
// Clear a resident adapter's device page table and rank (in `stream` order) and give its pages
// back to the free list in the order they were taken.
int drop_adapter(lora_pool* p, int32_t aid, lora_stream_t stream, const char* who) {
  if (!p->planning) {
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    if (p->ready_pending[aid]) e = cudaStreamWaitEvent(st, p->ev_ready[aid], 0);   // a packed load in flight
    if (e == cudaSuccess)
      e = cudaMemsetAsync(p->d_ptab + (size_t)aid * p->n_slots * kTabStride, 0xFF,
                          (size_t)p->n_slots * kTabStride * sizeof(int32_t), st);
    if (e == cudaSuccess) e = cudaMemsetAsync(p->d_rank + aid, 0, sizeof(int32_t), st);
    // loads that reuse these pages on other streams wait for this point of `st`
    if (e == cudaSuccess && !p->ev_freed) e = cudaEventCreateWithFlags(&p->ev_freed, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventRecord(p->ev_freed, st);
    if (e != cudaSuccess) return lora_cuda_fail(e, who);
    p->freed_recorded = true;
    p->ready_pending[aid] = 0;
  }
  int64_t n = 0;
  for (int32_t pg : p->tables[aid]) {
    if (pg < 0) continue;
    p->page_state[pg] = 0;
    p->free_list.push_back(pg);
    ++n;
  }
  p->adapter_pages -= n;
  p->rank[aid] = 0;
  p->refs[aid] = 0;
  p->tables[aid].clear();
  p->resident -= 1;
  return LORA_OK;
}

int64_t adapter_page_count(const lora_pool* p, int32_t aid) {
  int64_t n = 0;
  for (int32_t pg : p->tables[aid]) n += pg >= 0;
  return n;
}

// Idle resident adapters in eviction order (the pool's rule) and how many of them must go for
// `need` pages to be free; -1 if all of them would not be enough.
int evict_plan(const lora_pool* p, int64_t need, std::vector<int32_t>& order) {
  order.clear();
  for (int32_t a = 0; a < p->max_adapters; ++a)
    if (p->rank[a] != 0 && p->refs[a] == 0) order.push_back(a);
  if (p->evict_policy == LORA_EVICT_LRU) {
    std::sort(order.begin(), order.end(), [p](int32_t a, int32_t b) { return p->last_use[a] < p->last_use[b]; });
  } else if (p->evict_policy == LORA_EVICT_FARTHEST) {
    // next request of each idle adapter within the horizon; INT64_MAX = not requested there
    const int64_t horizon = p->lookahead > 0 ? std::min<int64_t>(p->lookahead, (int64_t)p->future.size())
                                             : (int64_t)p->future.size();
    std::vector<int64_t> nxt(p->max_adapters, INT64_MAX);
    for (int64_t i = horizon - 1; i >= 0; --i) {
      const int32_t a = p->future[i];
      if (a >= 0 && a < p->max_adapters) nxt[a] = i;
    }
    std::sort(order.begin(), order.end(), [p, &nxt](int32_t a, int32_t b) {
      if (nxt[a] != nxt[b]) return nxt[a] > nxt[b];    // farthest next request first
      return p->last_use[a] < p->last_use[b];          // not requested in the horizon: LRU
    });
  } else {
    std::sort(order.begin(), order.end(), [p](int32_t a, int32_t b) { return p->load_seq[a] < p->load_seq[b]; });
  }
  int64_t free_pages = (int64_t)p->free_list.size();
  int k = 0;
  while (free_pages < need && k < (int)order.size()) free_pages += adapter_page_count(p, order[k++]);
  return free_pages >= need ? k : -1;
}

int evict_idle(lora_pool* p, int64_t need, lora_stream_t stream, int32_t* evicted_host, int32_t* n_evicted,
               const char* who) {
  if (n_evicted) *n_evicted = 0;
  std::vector<int32_t> order;
  const int k = evict_plan(p, need, order);
  if (k < 0)
    return lora_fail(LORA_ENOPAGES, std::string(who) + ": " + std::to_string(need) + " pages needed, " +
                                        std::to_string(p->free_list.size()) + " free and idle adapters hold too few");
  for (int i = 0; i < k; ++i) {
    const int rc = drop_adapter(p, order[i], stream, who);
    if (rc != LORA_OK) return rc;
    if (evicted_host) evicted_host[i] = order[i];
    if (n_evicted) *n_evicted = i + 1;
  }
  return LORA_OK;
}
}  // namespace

extern "C" {

int lora_adapter_unload(lora_pool* p, int32_t aid, lora_stream_t stream) {
  if (!p) return lora_fail(LORA_EINVAL, "lora_adapter_unload: pool is NULL");
  if (aid < 0 || aid >= p->max_adapters || p->rank[aid] == 0)
    return lora_fail(LORA_EUNKNOWN_ADAPTER, "lora_adapter_unload: adapter " + std::to_string(aid) + " is not loaded");
  if (p->refs[aid] > 0)
    return lora_fail(LORA_EBUSY, "lora_adapter_unload: adapter " + std::to_string(aid) + " has " +
                                     std::to_string(p->refs[aid]) + " active requests");
  return drop_adapter(p, aid, stream, "lora_adapter_unload");
}

int lora_adapter_acquire(lora_pool* p, int32_t aid) {
  if (!p) return lora_fail(LORA_EINVAL, "lora_adapter_acquire: pool is NULL");
  if (aid < 0 || aid >= p->max_adapters || p->rank[aid] == 0)
    return lora_fail(LORA_EUNKNOWN_ADAPTER, "lora_adapter_acquire: adapter " + std::to_string(aid) + " is not loaded");
  p->refs[aid] += 1;
  p->last_use[aid] = ++p->use_clock;
  return LORA_OK;
}

int lora_pool_set_eviction(lora_pool* p, int32_t policy, const int32_t* future, int64_t n_future, int32_t lookahead) {
  if (!p || n_future < 0 || (n_future > 0 && !future) ||
      (policy != LORA_EVICT_LOAD_ORDER && policy != LORA_EVICT_LRU && policy != LORA_EVICT_FARTHEST))
    return lora_fail(LORA_EINVAL, "lora_pool_set_eviction: bad arguments");
  p->evict_policy = policy;
  p->future.assign(future, future + n_future);
  p->lookahead = lookahead;
  return LORA_OK;
}

int lora_adapter_release(lora_pool* p, int32_t aid) {
  if (!p) return lora_fail(LORA_EINVAL, "lora_adapter_release: pool is NULL");
  if (aid < 0 || aid >= p->max_adapters || p->rank[aid] == 0)
    return lora_fail(LORA_EUNKNOWN_ADAPTER, "lora_adapter_release: adapter " + std::to_string(aid) + " is not loaded");
  if (p->refs[aid] == 0)
    return lora_fail(LORA_EINVAL, "lora_adapter_release: adapter " + std::to_string(aid) + " has no active request");
  p->refs[aid] -= 1;
  return LORA_OK;
}

int32_t lora_adapter_refs(const lora_pool* p, int32_t aid) {
  if (!p || aid < 0 || aid >= p->max_adapters || p->rank[aid] == 0) return -1;
  return p->refs[aid];
}

int64_t lora_adapter_packed_size(const lora_pool* p, int32_t rank, const int32_t* present) {
  if (!p || rank < 1 || rank > LORA_MAX_RANK) return (int64_t)lora_fail(LORA_EINVAL, "lora_adapter_packed_size: bad arguments");
  int64_t n_present = 0;
  for (int s = 0; s < p->n_slots; ++s) n_present += (!present || present[s] != 0);
  return (int64_t)packed_layout(p, rank, n_present).total;
}

int lora_adapter_pack(const lora_pool* p, int32_t rank, const void* const* A_host, const void* const* B_host,
                      void* packed, int64_t packed_bytes) {
  if (!p || rank < 1 || rank > LORA_MAX_RANK || !A_host || !B_host || !packed)
    return lora_fail(LORA_EINVAL, "lora_adapter_pack: bad arguments");
  int64_t n_present = 0;
  for (int s = 0; s < p->n_slots; ++s) {
    if (!A_host[s]) continue;
    if (!B_host[s]) return lora_fail(LORA_EINVAL, "lora_adapter_pack: B_host[slot] is NULL where A_host[slot] is set");
    ++n_present;
  }
  const PackedLayout PL = packed_layout(p, rank, n_present);
  if (packed_bytes < (int64_t)PL.total)
    return lora_fail(LORA_EINVAL, "lora_adapter_pack: buffer has " + std::to_string(packed_bytes) + " bytes, needs " +
                                      std::to_string(PL.total));
  const int64_t H = p->H;
  uint16_t* rows = reinterpret_cast<uint16_t*>(static_cast<char*>(packed) + PL.rows);
  std::vector<uint8_t> present(p->n_slots);
  for (int s = 0; s < p->n_slots; ++s) present[s] = A_host[s] != nullptr;
  pack_rows(A_host, B_host, present, H, rank, rows);
  return LORA_OK;
}

int lora_adapter_load_packed(lora_pool* p, int32_t aid, int32_t rank, const int32_t* present, const void* packed,
                             int64_t packed_bytes, lora_stream_t copy_stream, int32_t* table_out) {
  if (!p) return lora_fail(LORA_EINVAL, "lora_adapter_load_packed: pool is NULL");
  if (p->planning) return lora_fail(LORA_EINVAL, "lora_adapter_load_packed: planning pool has no device state");
  if (aid < 0 || aid >= p->max_adapters)
    return lora_fail(LORA_EINVAL, "lora_adapter_load_packed: adapter id " + std::to_string(aid) + " outside [0, max_adapters)");
  if (rank < 1 || rank > LORA_MAX_RANK)
    return lora_fail(LORA_ERANK, "lora_adapter_load_packed: rank " + std::to_string(rank) + " outside [1, 64]");
  if (p->rank[aid] != 0)
    return lora_fail(LORA_EEXIST, "lora_adapter_load_packed: adapter " + std::to_string(aid) + " already loaded");
  if (!packed || (reinterpret_cast<uintptr_t>(packed) & 15) != 0)
    return lora_fail(LORA_EINVAL, "lora_adapter_load_packed: packed buffer must be 16-byte aligned");
  const int S = p->n_slots;
  int64_t n_present = 0;
  for (int s = 0; s < S; ++s) n_present += (!present || present[s] != 0);
  const PackedLayout PL = packed_layout(p, rank, n_present);
  if (packed_bytes < (int64_t)PL.total)
    return lora_fail(LORA_EINVAL, "lora_adapter_load_packed: buffer has " + std::to_string(packed_bytes) +
                                      " bytes, needs " + std::to_string(PL.total));
  void* dptr = nullptr;
  if (cudaHostGetDevicePointer(&dptr, const_cast<void*>(packed), 0) != cudaSuccess || !dptr) {
    cudaGetLastError();
    return lora_fail(LORA_EINVAL, "lora_adapter_load_packed: packed buffer is not pinned host memory");
  }
  if (PL.need > (int64_t)p->free_list.size())
    return lora_fail(LORA_ENOPAGES, "lora_adapter_load_packed: adapter needs " + std::to_string(PL.need) + " pages, " +
                                        std::to_string(p->free_list.size()) + " free");
  // Take pages as lora_adapter_load does and write the header the kernel reads.
  char* host = static_cast<char*>(const_cast<void*>(packed));
  int32_t* ids = reinterpret_cast<int32_t*>(host + PL.ids);
  int32_t* tab_image = reinterpret_cast<int32_t*>(host + PL.tab);
  std::vector<int32_t> table((size_t)S * 2 * rank, -1);
  std::vector<int32_t> taken;
  taken.reserve(PL.need);
  for (int i = 0; i < S * kTabStride; ++i) tab_image[i] = -1;
  for (int s = 0; s < S; ++s) {
    if (present && present[s] == 0) continue;
    for (int half = 0; half < 2; ++half)
      for (int j = 0; j < rank; ++j) {
        const int32_t pg = p->free_list.back();
        p->free_list.pop_back();
        table[((size_t)s * 2 + half) * rank + j] = pg;
        tab_image[s * kTabStride + half * LORA_MAX_RANK + j] = pg;
        ids[taken.size()] = pg;
        taken.push_back(pg);
      }
  }
  cudaStream_t st = reinterpret_cast<cudaStream_t>(copy_stream);
  cudaError_t e = cudaSuccess;
  if (p->freed_recorded) e = cudaStreamWaitEvent(st, p->ev_freed, 0);      // reused pages are no longer read
  if (e == cudaSuccess && !p->ev_ready[aid]) e = cudaEventCreateWithFlags(&p->ev_ready[aid], cudaEventDisableTiming);
  if (e == cudaSuccess) {
    ProfScope prof(p, LORA_KIND_SCATTER, st);
    const char* dbase = static_cast<const char*>(dptr);
    const int grid = (int)std::min<int64_t>(std::max<int64_t>(PL.need, 1), 4 * (int64_t)device_sm_count());
    load_packed_kernel<<<grid, 256, 0, st>>>(reinterpret_cast<const int32_t*>(dbase + PL.ids),
                                              reinterpret_cast<const int32_t*>(dbase + PL.tab),
                                              reinterpret_cast<const uint4*>(dbase + PL.rows), PL.need, p->H,
                                              reinterpret_cast<uint4*>(p->pool_dev),
                                              p->d_ptab + (size_t)aid * S * kTabStride, S * kTabStride, p->d_rank + aid,
                                              rank);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) e = cudaEventRecord(p->ev_ready[aid], st);
  if (e != cudaSuccess) {
    for (auto it = taken.rbegin(); it != taken.rend(); ++it) p->free_list.push_back(*it);
    return lora_cuda_fail(e, "lora_adapter_load_packed");
  }
  for (int32_t pg : taken) p->page_state[pg] = 2;
  p->rank[aid] = rank;
  p->refs[aid] = 0;
  p->load_seq[aid] = p->next_seq++;
  p->last_use[aid] = ++p->use_clock;
  p->tables[aid] = table;
  p->adapter_pages += PL.need;
  p->resident += 1;
  p->ready_pending[aid] = 1;
  if (table_out) std::memcpy(table_out, table.data(), table.size() * sizeof(int32_t));
  return LORA_OK;
}

int lora_adapter_wait(lora_pool* p, int32_t aid, lora_stream_t stream) {
  if (!p) return lora_fail(LORA_EINVAL, "lora_adapter_wait: pool is NULL");
  if (aid < 0 || aid >= p->max_adapters || p->rank[aid] == 0)
    return lora_fail(LORA_EUNKNOWN_ADAPTER, "lora_adapter_wait: adapter " + std::to_string(aid) + " is not loaded");
  if (p->planning || !p->ready_pending[aid]) return LORA_OK;
  cudaError_t e = cudaStreamWaitEvent(reinterpret_cast<cudaStream_t>(stream), p->ev_ready[aid], 0);
  return e == cudaSuccess ? LORA_OK : lora_cuda_fail(e, "lora_adapter_wait");
}

int lora_pool_evict_idle(lora_pool* p, int64_t need, lora_stream_t stream, int32_t* evicted_host, int32_t* n_evicted) {
  if (n_evicted) *n_evicted = 0;
  if (!p || need < 0) return lora_fail(LORA_EINVAL, "lora_pool_evict_idle: bad arguments");
  return evict_idle(p, need, stream, evicted_host, n_evicted, "lora_pool_evict_idle");
}

int lora_adapter_ensure(lora_pool* p, int32_t aid, int32_t rank, const void* const* A_host, const void* const* B_host,
                        lora_stream_t stream, int32_t* table_out, int32_t* loaded_out, int32_t* evicted_host,
                        int32_t* n_evicted) {
  if (loaded_out) *loaded_out = 0;
  if (n_evicted) *n_evicted = 0;
  if (!p) return lora_fail(LORA_EINVAL, "lora_adapter_ensure: pool is NULL");
  if (aid < 0 || aid >= p->max_adapters)
    return lora_fail(LORA_EINVAL, "lora_adapter_ensure: adapter id " + std::to_string(aid) + " outside [0, max_adapters)");
  if (p->rank[aid] != 0) {                       // resident: one more active request
    if (rank != p->rank[aid])
      return lora_fail(LORA_ERANK, "lora_adapter_ensure: adapter " + std::to_string(aid) + " is resident with rank " +
                                       std::to_string(p->rank[aid]));
    p->refs[aid] += 1;
    p->last_use[aid] = ++p->use_clock;
    if (table_out) std::memcpy(table_out, p->tables[aid].data(), p->tables[aid].size() * sizeof(int32_t));
    return LORA_OK;
  }
  if (rank < 1 || rank > LORA_MAX_RANK)
    return lora_fail(LORA_ERANK, "lora_adapter_ensure: rank " + std::to_string(rank) + " outside [1, 64]");
  if (!p->planning && (!A_host || !B_host))
    return lora_fail(LORA_EINVAL, "lora_adapter_ensure: A_host and B_host arrays are required");
  if (!p->planning)                              // argument errors are found before anything is evicted
    for (int s = 0; s < p->n_slots; ++s)
      if (A_host[s] && !B_host[s]) return lora_fail(LORA_EINVAL, "lora_adapter_ensure: B_host[slot] is NULL where A_host[slot] is set");
  int64_t n_present = 0;
  for (int s = 0; s < p->n_slots; ++s) n_present += (A_host == nullptr || A_host[s] != nullptr);
  const int64_t need = 2 * (int64_t)rank * n_present;
  int rc = evict_idle(p, need, stream, evicted_host, n_evicted, "lora_adapter_ensure");
  if (rc != LORA_OK) return rc;
  rc = lora_adapter_load(p, aid, rank, A_host, B_host, stream, table_out);
  if (rc != LORA_OK) return rc;
  p->refs[aid] = 1;
  if (loaded_out) *loaded_out = 1;
  return LORA_OK;
}

void lora_pool_stats(const lora_pool* p, lora_pool_stats_t* out) {
  if (!p || !out) return;
  out->num_pages = p->num_pages;
  out->free_pages = (int64_t)p->free_list.size();
  out->adapter_pages = p->adapter_pages;
  out->reserved_pages = p->reserved_pages;
  out->resident_adapters = p->resident;
  out->max_adapters = p->max_adapters;
}

int lora_status(lora_pool* p, lora_stream_t stream) {
  if (!p) return lora_fail(LORA_EINVAL, "lora_status: pool is NULL");
  if (p->planning) return LORA_OK;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int32_t h[4] = {0, 0, 0, 0};
  cudaError_t e = cudaMemcpyAsync(h, p->d_err, sizeof(h), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e == cudaSuccess) e = cudaMemsetAsync(p->d_err, 0, sizeof(h), st);
  if (e != cudaSuccess) return lora_cuda_fail(e, "lora_status");
  if (h[0] == 0) return LORA_OK;
  std::string msg = "device check failed:";
  if (h[1] & LORA_DEV_UNKNOWN_ADAPTER) msg += " unknown adapter id in token_adapter;";
  if (h[1] & LORA_DEV_BAD_PAGE) msg += " page id out of range;";
  if (h[1] & LORA_DEV_BAD_RANK) msg += " rank out of range;";
  if (h[1] & LORA_DEV_WAIT_TIMEOUT) msg += " a bounded wait ran out;";
  if (h[1] & LORA_DEV_BAD_SEGMENT) msg += " inconsistent segment list;";
  return lora_fail(LORA_EDEVICE, msg);
}

// ---- segment workspace -----------------------------------------------------------------
namespace {
SegLayout seg_layout(const lora_pool* p, int32_t T_max, int32_t max_group) {
  return segments_layout(T_max, p->H, p->max_adapters, max_group);
}
}  // namespace

int64_t lora_segments_size_group(const lora_pool* p, int32_t T_max, int32_t max_group) {
  if (!p || T_max < 1 || T_max > LORA_MAX_TOKENS || max_group < 1 || max_group > LORA_MAX_GROUP)
    return (int64_t)lora_fail(LORA_EINVAL, "lora_segments_size: bad arguments");
  return (int64_t)seg_layout(p, T_max, max_group).total;
}

int64_t lora_segments_size(const lora_pool* p, int32_t T_max) { return lora_segments_size_group(p, T_max, 1); }

int lora_segments_init_group(const lora_pool* p, void* ws, int64_t ws_bytes, int32_t T_max, int32_t max_group,
                             lora_segments* seg) {
  if (!p || !ws || !seg || T_max < 1 || T_max > LORA_MAX_TOKENS || max_group < 1 || max_group > LORA_MAX_GROUP)
    return lora_fail(LORA_EINVAL, "lora_segments_init: bad arguments");
  if ((reinterpret_cast<uintptr_t>(ws) & 255) != 0)
    return lora_fail(LORA_EINVAL, "lora_segments_init: workspace must be 256-byte aligned");
  const SegLayout L = seg_layout(p, T_max, max_group);
  if (ws_bytes < (int64_t)L.total)
    return lora_fail(LORA_EINVAL, "lora_segments_init: workspace has " + std::to_string(ws_bytes) + " bytes, needs " +
                                      std::to_string(L.total));
  char* b = static_cast<char*>(ws);
  seg->T_max = T_max;
  seg->T = -1;
  seg->max_seg = L.max_seg;
  seg->H = p->H;
  seg->perm = reinterpret_cast<int32_t*>(b + L.perm);
  seg->seg_off = reinterpret_cast<int32_t*>(b + L.seg_off);
  seg->seg_adapter = reinterpret_cast<int32_t*>(b + L.seg_adapter);
  seg->n_seg = reinterpret_cast<int32_t*>(b + L.n_seg);
  seg->tok_adapter = reinterpret_cast<int32_t*>(b + L.tok_adapter);
  seg->units = reinterpret_cast<int32_t*>(b + L.units);
  seg->n_units = reinterpret_cast<int32_t*>(b + L.n_units);
  seg->unit_cap = L.unit_cap;
  seg->delta_slots = max_group;
  seg->delta = reinterpret_cast<float*>(b + L.delta);
  seg->gemm_partials = reinterpret_cast<float*>(b + L.partials);
  const bool fused = L.n_tiles_max > 0;
  seg->n_tiles_max = L.n_tiles_max;
  seg->tile_plan = fused ? reinterpret_cast<int32_t*>(b + L.tile_plan) : nullptr;
  seg->entries = fused ? reinterpret_cast<int32_t*>(b + L.entries) : nullptr;
  seg->n_entries = fused ? reinterpret_cast<int32_t*>(b + L.n_entries) : nullptr;
  seg->units_rest = fused ? reinterpret_cast<int32_t*>(b + L.units_rest) : nullptr;
  seg->n_units_rest = fused ? reinterpret_cast<int32_t*>(b + L.n_units_rest) : nullptr;
  seg->s_lora = fused ? reinterpret_cast<uint16_t*>(b + L.s_lora) : nullptr;
  seg->shrink_scratch = fused ? reinterpret_cast<float*>(b + L.shrink_scratch) : nullptr;
  return LORA_OK;
}

int lora_segments_init(const lora_pool* p, void* ws, int64_t ws_bytes, int32_t T_max, lora_segments* seg) {
  return lora_segments_init_group(p, ws, ws_bytes, T_max, 1, seg);
}

}  // extern "C"
