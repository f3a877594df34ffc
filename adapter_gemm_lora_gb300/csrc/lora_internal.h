// Internal declarations shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <string>
#include <unordered_map>
#include <vector>

#include "../../include/lora.h"

// Device error word layout (int32[4]): [0] first error code (LORA_E*), [1] detail bits.
enum : int32_t {
  LORA_DEV_UNKNOWN_ADAPTER = 1 << 0,   // token id out of range or not loaded
  LORA_DEV_BAD_PAGE = 1 << 1,          // page id outside [0, num_pages)
  LORA_DEV_BAD_RANK = 1 << 2,          // rank outside [1, 64]
  LORA_DEV_WAIT_TIMEOUT = 1 << 3,      // a bounded mbarrier wait gave up
  LORA_DEV_BAD_SEGMENT = 1 << 4,       // inconsistent segment / work list
};

// Page table entries per (adapter, slot): [2][LORA_MAX_RANK] int32.
constexpr int kTabStride = 2 * LORA_MAX_RANK;
// Work-list geometry shared by the segment builder and the gather kernels.
constexpr int kUnitTokens = 16;      // tokens per LoRA-delta work unit
constexpr int kUnitMixed = 1 << 8;   // in units_rest: the unit also holds tokens of fused tiles

struct lora_pool {
  void* pool_dev = nullptr;
  int64_t num_pages = 0;
  int32_t H = 0;
  int32_t n_slots = 0;
  int32_t max_adapters = 0;
  bool planning = false;
  int device = -1;

  // host bookkeeping
  std::vector<int32_t> free_list;                 // taken from the back
  std::vector<uint8_t> page_state;                // 0 free, 1 reserved, 2 adapter, 4 KV of a request
  std::vector<int32_t> rank;                      // per adapter id; 0 = not loaded
  std::vector<std::vector<int32_t>> tables;       // per adapter id: [n_slots][2][rank]
  std::vector<int32_t> refs;                      // per adapter id: active requests
  std::vector<int64_t> load_seq;                  // per adapter id: order of its load
  int64_t next_seq = 0;
  std::vector<int64_t> last_use;                  // per adapter id: clock of its last load / ensure / acquire
  int64_t use_clock = 0;
  int32_t evict_policy = LORA_EVICT_LOAD_ORDER;   // which idle adapter goes first
  std::vector<cudaEvent_t> ev_ready;              // per adapter id: completion of its last packed load
  std::vector<uint8_t> ready_pending;             // per adapter id: that load may still be in flight
  cudaEvent_t ev_freed = nullptr;                 // recorded after every unload / eviction
  bool freed_recorded = false;
  struct KVReq {
    int32_t layers = 0;
    std::vector<int32_t> pages;                   // per token: per layer, K page then V page
  };
  std::unordered_map<int64_t, KVReq> kv;          // request id -> its KV pages
  std::vector<int32_t> h_kvtab;                   // host staging of lora_kv_batch_table
  std::vector<int32_t> future;                    // upcoming adapter requests (farthest-future rule)
  int32_t lookahead = 0;                          // entries of `future` looked at; <= 0: all
  int64_t adapter_pages = 0;
  int64_t reserved_pages = 0;
  int32_t resident = 0;

  // device state owned by the library
  int32_t* d_ptab = nullptr;    // [max_adapters][n_slots][2][64]
  int32_t* d_rank = nullptr;    // [max_adapters]
  int32_t* d_err = nullptr;     // [4]
  void* d_stage = nullptr;      // staging area for adapter loads
  size_t d_stage_bytes = 0;
  std::vector<uint16_t> h_stage;

  // kernel accounting (lora_profile_*)
  int64_t launches[LORA_N_KINDS] = {};
  bool prof_on = false;
  struct ProfRec { int kind; cudaEvent_t start, stop; };
  std::vector<ProfRec> prof_rec;
  std::vector<cudaEvent_t> ev_free;
};

// Bracket one kernel launch: count it and, when profiling is on, record events around it.
struct ProfScope {
  lora_pool* p;
  int kind;
  cudaStream_t st;
  int rec = -1;
  bool capturing = false;
  ProfScope(const lora_pool* pool, int k, cudaStream_t s);
  ~ProfScope();
};

// Error reporting (thread-local message).
int lora_fail(int code, const std::string& msg);
int lora_cuda_fail(cudaError_t e, const char* what);

// Kernel launchers (return LORA_OK or LORA_ECUDA).
int launch_scatter_pages(const uint16_t* stage, const int32_t* d_pages, int64_t n_pages, int32_t H,
                         void* pool_dev, cudaStream_t st);
int launch_segments_build(const lora_pool* pool, const int32_t* token_adapter, int32_t T,
                          const lora_segments* seg, cudaStream_t st, bool pdl);

// One LoRA-delta launch covers n_group projection slots that read the same input x (the q, k
// and v projections of a layer): every work unit is done once per slot, with that slot's page
// table, into that slot's delta buffer.
struct LoraLaunch {
  const uint16_t* pool;
  int64_t num_pages;
  int32_t H, T, n_slots;
  int32_t n_group;                     // 1 .. LORA_MAX_GROUP
  int32_t slot[LORA_MAX_GROUP];
  float* delta[LORA_MAX_GROUP];        // [T][H] fp32 per slot of the group
  const int32_t* ptab;
  const int32_t* rank;
  const lora_segments* seg;
  const int32_t* units;                // the work list: seg->units, or seg->units_rest when the
  const int32_t* n_units;              // fused tiles take their LoRA term in the GEMM
  const int32_t* tile_plan;            // non-null: tokens of fused tiles are skipped
  const uint16_t* x;
  int32_t* err;
  bool pdl;
};
int launch_lora_delta(const LoraLaunch& L, cudaStream_t st);

// Shrink of the fused tiles (s = x A, for every group member of the call) into seg->s_lora.
struct ShrinkLaunch {
  const uint16_t* pool;
  int64_t num_pages;
  int32_t H, T, n_slots;
  int32_t n_group;
  int32_t slot[LORA_MAX_GROUP];
  const int32_t* ptab;
  const int32_t* rank;
  const lora_segments* seg;
  const uint16_t* x;
  int32_t* err;
  bool pdl;
};
int launch_lora_shrink(const ShrinkLaunch& S, cudaStream_t st);

struct GemmLaunch {
  const uint16_t* x;       // [T][H]
  const uint16_t* W;       // [H][H] (out, in)
  uint16_t* y;             // [T][H]
  const float* delta;      // [T][H]
  const int32_t* tok_adapter;  // [T] validated ids
  const int32_t* ptab;
  float* partials;         // split-K scratch (batches of <= 256 tokens)
  int64_t partials_floats; // its capacity; the split is used only when it fits
  int32_t T, H, slot, n_slots;
  int32_t* err;
  bool pdl;
  // fused tiles of a prefill-shaped batch (launch_gemm_fused)
  const int32_t* tile_plan;
  const uint16_t* s_lora;  // [T][kSCols] bf16, this slot's s of the fused tiles
  const uint16_t* pool;
  int64_t num_pages;
  const int32_t* rank;
  float* lora_dbg;         // the LoRA-only launch writes the fp32 LoRA term of the fused tiles here
  const lora_pool* prof;   // each kernel launch is one profiling scope of kind gemm on this pool
};
int launch_gemm(const GemmLaunch& G, cudaStream_t st);
// n (1 .. LORA_MAX_GROUP) slots that read the same x whose batch is cut into 256-token tiles on
// the persistent GEMM: the fused tiles of the plan take their LoRA term inside the GEMM.
// gemm_fused_fits says whether the geometry allows it; lora_only runs only that term, into
// G[i].lora_dbg, for the fused tiles.
bool gemm_fused_fits(const GemmLaunch* G, int n);
int launch_gemm_fused(const GemmLaunch* G, int n, bool lora_only, cudaStream_t st);
// n (2 .. LORA_MAX_GROUP) slots that read the same x, batches of <= 256 tokens: one persistent
// split-K launch over every (slot, feature tile).  gemm_group_fits says whether the group
// qualifies (split-K geometry, one x, scratch for n slots); otherwise launch_gemm per slot.
bool gemm_group_fits(const GemmLaunch* G, int n);
int launch_gemm_group(const GemmLaunch* G, int n, cudaStream_t st);
// Capacity of the base GEMM's split-K scratch for a workspace of T_max tokens: 3 partial tiles
// (4-way split) of up to 256 token columns, the tile rounded up to 128 columns.
constexpr int64_t gemm_partial_floats(int32_t T_max, int32_t H) {
  return 3 * (((T_max < 256 ? T_max : 256) + 127) / 128 * 128) * (int64_t)H;
}

// Byte offsets of the arrays of a segment workspace (lora_segments_init) for batches of up to
// T_max tokens, hidden size H, adapter ids below max_adapters and group calls of up to
// max_group slots; every array starts on a 256-byte boundary.
// Fused tiles of prefill-shaped batches: tiles of 256 tokens with at most 4 adapters, whose
// LoRA term the base GEMM adds from s = x A (bf16 hi and lo parts, 512 columns per token: tile
// slot b's hi part in [128 b, 128 b + 64), its lo part in [128 b + 64, 128 b + 128)).
constexpr int kTileTokens = LORA_TILE_TOKENS;
constexpr int kTileAdapters = LORA_TILE_ADAPTERS;
constexpr int kPlanStride = 8;                         // int32 per tile in tile_plan
constexpr int kSCols = 2 * LORA_MAX_RANK * kTileAdapters;   // bf16 columns of s_lora per token
// The shrink kernel's persistent clusters (4 CTAs, one K quarter each) exchange partial sums of
// s through global scratch: per cluster and item parity, 4 owners x 3 senders x [64 tokens][128
// rows] fp32.
constexpr int kShrinkCluster = 4;
constexpr int kShrinkMaxClusters = 40;
constexpr size_t kShrinkScratchFloats =
    (size_t)kShrinkMaxClusters * 2 * kShrinkCluster * (kShrinkCluster - 1) * 64 * 128;
constexpr int32_t fused_tiles_max(int32_t T_max) { return T_max > kTileTokens ? (T_max + kTileTokens - 1) / kTileTokens : 0; }

struct SegLayout {
  size_t perm, seg_off, seg_adapter, n_seg, tok_adapter, units, n_units, delta, partials;
  size_t tile_plan, entries, n_entries, units_rest, n_units_rest, s_lora, shrink_scratch, total;
  int32_t max_seg, unit_cap, n_tiles_max;
};
constexpr size_t align256(size_t v) { return (v + 255) / 256 * 256; }
constexpr SegLayout segments_layout(int32_t T_max, int32_t H, int32_t max_adapters, int32_t max_group) {
  SegLayout L{};
  L.max_seg = T_max < max_adapters ? T_max : max_adapters;
  L.unit_cap = T_max / kUnitTokens + L.max_seg + 1;
  L.n_tiles_max = fused_tiles_max(T_max);
  const bool fused = L.n_tiles_max > 0;
  size_t off = 0;
  L.perm = off;         off = align256(off + (size_t)T_max * 4);
  L.seg_off = off;      off = align256(off + (size_t)(L.max_seg + 2) * 4);
  L.seg_adapter = off;  off = align256(off + (size_t)(L.max_seg + 1) * 4);
  L.n_seg = off;        off = align256(off + 16);
  L.tok_adapter = off;  off = align256(off + (size_t)T_max * 4);
  L.units = off;        off = align256(off + (size_t)L.unit_cap * 16);
  L.n_units = off;      off = align256(off + 16);
  L.delta = off;        off = align256(off + (size_t)max_group * T_max * H * 4);
  L.partials = off;     off = align256(off + (size_t)max_group * gemm_partial_floats(T_max, H) * 4);
  L.tile_plan = off;    off = align256(off + (size_t)L.n_tiles_max * kPlanStride * 4);
  L.entries = off;      off = align256(off + (size_t)L.n_tiles_max * kTileAdapters * 4);
  L.n_entries = off;    off = align256(off + (fused ? 16 : 0));
  L.units_rest = off;   off = align256(off + (fused ? (size_t)L.unit_cap * 16 : 0));
  L.n_units_rest = off; off = align256(off + (fused ? 16 : 0));
  L.s_lora = off;       off = align256(off + (fused ? (size_t)max_group * T_max * kSCols * 2 : 0));
  L.shrink_scratch = off; off = align256(off + (fused ? kShrinkScratchFloats * 4 : 0));
  L.total = off;
  return L;
}

// Programmatic dependent launch: every kernel of the path waits for the kernel before it
// (griddepcontrol.wait) before touching anything an earlier kernel writes, and only then
// lets its own dependent start (griddepcontrol.launch_dependents).  So when a kernel starts,
// the kernel two places before it has completed, and launch latency and prologues overlap.
__device__ __forceinline__ void pdl_wait_then_release() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Launch `kernel` on `st`, as a programmatic dependent of the previous kernel in the stream
// when `pdl` is set.  (With per-kernel profiling events recorded between kernels the overlap
// cannot happen anyway, and such launches are made without the attribute.)
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(bool pdl, void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

int device_sm_count();

// Kernel attributes are per device: each launcher keeps one flag per device ordinal saying that
// its kernel's dynamic shared-memory limit has been raised there.  Setting an attribute twice is
// harmless, so two host threads racing on a first launch both just set it.
constexpr int kMaxDeviceFlags = 64;
struct DeviceFlags {
  std::atomic<bool> set[kMaxDeviceFlags] = {};
};
template <typename Kernel>
int ensure_smem_attr(DeviceFlags& flags, Kernel* kernel, int bytes, const char* what) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return lora_cuda_fail(e, what);
  const bool cached = dev >= 0 && dev < kMaxDeviceFlags;
  if (cached && flags.set[dev].load(std::memory_order_acquire)) return LORA_OK;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return lora_cuda_fail(e, what);
  if (cached) flags.set[dev].store(true, std::memory_order_release);
  return LORA_OK;
}

