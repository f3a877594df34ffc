// The LoRA delta of one projection slot: the two skinny products of the unmerged term.
//
// "S-LoRA, in depth", section "Merge or keep adapters separate": besides the shared xW,
// each token needs (xA)B for its own adapter.  Section "Kernels for a batch of mixed ranks":
// A and B sit in scattered pool pages and ranks differ inside one batch, so both products
// gather their operands through the page table.  Here they run fused in one kernel:
//   shrink  s[t, j]     = sum_k x[t, k] * A[k, j]        (A page j = column j of A, H values)
//   expand  delta[t, n] = sum_j s[t, j] * B[j, n]        (B page j = row j of B, H values)
//
// Work unit: up to 16 tokens of one segment (tokens that share an adapter), handled by a
// cluster of KC CTAs (KC = 2 for H <= 2048, else 4).
// One launch may serve several projection slots that read the same x (q, k and v of a layer):
// its work items are then every unit once per slot, each with its slot's page table and delta
// buffer, so the short per-slot work lists of a decode batch become one list long enough to keep
// every cluster busy.  CTA q owns one share of the feature range, [q H/KC, (q+1) H/KC), for both
// products: it reads that share of the unit's token rows of x, of all r A pages and of all r B
// pages, and nothing else.  The shrink over its share gives partial sums of s; the KC partials
// are exchanged through distributed shared memory and added in cluster-rank order, so every CTA
// holds the same complete s.  The expand then writes the CTA's share of delta.
//
// Data movement: one producer warp streams page-row slices with TMA bulk copies (cp.async.bulk):
// the unit's x rows into a buffer of their own, held across the shrink, and the A pages, then the
// B pages, into a ring of stages, each lane copying one row.  Feature blocks of 1024 (2 KB
// slices): 2 stages of 32 rows (two groups of 16 rank columns).  A CTA share of 1280 features
// (H = 5120, 4 CTAs) is one block of 2.5 KB slices instead of 1024 + 256: 3 stages of 16 rows.
// The x buffer and the ring take the same shared memory either way.
// Eight consumer warps multiply what has landed on the tensor cores with the warp-level bf16 MMA
// (m16n8k16, fp32 accumulation), feeding operands with ldmatrix straight from the staged page
// rows: a unit holds 16 tokens at most, below the 64-row minimum tile of the asynchronous
// tcgen05 MMA, while ldmatrix takes any row addresses, which is what a page gather produces.
// The MMAs exist only to keep the 16-way reuse of every loaded byte off the CUDA cores; the
// kernel is bound by moving the bytes it gathers, through a fixed chain per item (x rows,
// shrink, exchange, expand, stores).
//
// Precision: bf16 inputs, exact products, fp32 accumulation.  s is passed to the expand as
// two bf16 terms (s = hi + lo, with hi = bf16(s), lo = bf16(s - hi)), which keeps 16 bits of
// its mantissa.  The order of every sum is fixed and depends neither on page placement nor on
// the other tokens of the batch.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "lora_internal.h"

namespace {

constexpr int kUnitTok = kUnitTokens;         // tokens per unit (16)
constexpr int kXRows = kUnitTok;               // x rows of the unit: a buffer of their own
constexpr int kConsumerWarps = 8;
constexpr int kConsumers = 32 * kConsumerWarps;
constexpr int kThreads = kConsumers + 32;      // + one producer warp
constexpr int kSbPitch = LORA_MAX_RANK + 8;    // bf16 elements per token row of s (hi or lo)
constexpr int kMaxStages = 3;
// Ring geometry for feature blocks of FBW features.  Staged rows are padded by 16 bytes so that
// the 8 rows an ldmatrix phase reads fall in 8 different 16-byte bank groups.
template <int FBW>
struct Ring {
  static constexpr int kGroups = FBW > 1024 ? 1 : 2;          // groups of 16 rank columns a stage
  static constexpr int kRows = 16 * kGroups;                  // page rows per stage
  static constexpr int kRowBytes = FBW * 2 + 16;
  static constexpr int kSlotBytes = kRows * kRowBytes;
  static constexpr int kStages = FBW > 1024 ? 3 : 2;
  static constexpr int kOffX = kStages * kSlotBytes;          // [16 tokens][kRowBytes] after the ring
  static constexpr int kMT = FBW / 16 / kConsumerWarps;       // expand: 16-feature tiles per warp
  static_assert(kStages <= kMaxStages && FBW % (16 * kConsumerWarps) == 0, "ring geometry");
};
// shared memory layout (dynamic): the ring and the x buffer in one area, then the rest
constexpr int kAreaBytes = Ring<1024>::kOffX + kXRows * Ring<1024>::kRowBytes;
static_assert(Ring<1280>::kOffX + kXRows * Ring<1280>::kRowBytes <= kAreaBytes, "ring area");
constexpr int kOffRing = 0;
constexpr int kOffPart = kAreaBytes;                                         // [8 warps][16][16] f32
static_assert(kUnitTok == 16, "the MMA tiling assumes 16 tokens per unit");
// The rest of the layout depends on the number KC of CTAs that split an item's features.
template <int KC>
struct Smem {
  static constexpr int kOffExch = kOffPart + kConsumerWarps * 16 * 16 * 4;                 // [2][KC][64][16] f32
  static constexpr int kOffSb = kOffExch + 2 * KC * LORA_MAX_RANK * kUnitTok * 4;          // [2][16][kSbPitch] bf16
  static constexpr int kOffBar = kOffSb + 2 * kUnitTok * kSbPitch * 2;
  static constexpr int kBytes = kOffBar + (2 * kMaxStages + 4) * 8;
  static_assert(kBytes <= 227 * 1024, "shared memory budget");
  static_assert(kOffSb % 16 == 0 && kOffBar % 8 == 0, "alignment");
};

__device__ __forceinline__ void flag_error(int32_t* err, int32_t bits) {
  atomicCAS(err, 0, LORA_EDEVICE);
  atomicOr(err + 1, bits);
}
__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

// ---- mbarriers, bulk copies, cluster -------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(1000000u)
      : "memory");
  return ok != 0;
}
// Bounded wait (about 2 s at the maximum SM clock, counted with the SM's cycle counter).
constexpr long long kWaitLimitCycles = 4000000000ll;
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long c0 = clock64();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (clock64() - c0 > kWaitLimitCycles) return false;
  }
}
// The same wait in every lane of a warp, with one warp-wide verdict.
__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity));
}
// Copy `bytes` (multiple of 16, both addresses 16-byte aligned) from global to this CTA's
// shared memory; completion is counted on `bar` as transaction bytes.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory"); }

// ---- warp-level MMA --------------------------------------------------------------------------
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
// D[16x8] += A[16x16] B[16x8], bf16 operands, fp32 accumulators.
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// One work item: a work unit as the segment builder wrote it, for one slot of the launch's
// group, plus the per-lane entries a warp gathers for it: the page ids of rank columns lane
// and lane + 32 (-1 past the rank) and perm entries.
struct Unit {
  int r, t_begin, n_tok;
  bool mixed;              // some of its tokens belong to fused tiles (skipped here)
  const int32_t* tab;      // the adapter's page table on the item's slot
  float* delta;            // the slot's delta rows
};
__device__ __forceinline__ int4 load_rec(const LoraLaunch& L, int u, int n_units) {
  return u < n_units ? __ldg(reinterpret_cast<const int4*>(L.units) + u) : make_int4(0, 0, 0, 0);
}
// Item i of the launch is unit i / n_group on group member i % n_group.
__device__ __forceinline__ Unit unit_of(const LoraLaunch& L, const int4& rec, int g) {
  Unit U;
  U.r = rec.y;
  U.t_begin = rec.z;
  U.n_tok = rec.w & (kUnitMixed - 1);
  U.mixed = (rec.w & kUnitMixed) != 0;
  int slot = L.slot[0];
  float* d = L.delta[0];
#pragma unroll
  for (int k = 1; k < LORA_MAX_GROUP; ++k)
    if (g == k) {
      slot = L.slot[k];
      d = L.delta[k];
    }
  U.tab = L.ptab + ((int64_t)rec.x * L.n_slots + slot) * kTabStride;
  U.delta = d;
  return U;
}
struct Gathered {
  int32_t pa[2], pb[2];
  int32_t tok[4];
};
// Issue this lane's loads for unit U (values are consumed one unit later).  ntok_lane: how many
// perm entries each lane reads; entry k of lane l is token tok_index(l, k) of the unit.  A token
// of a fused tile (its LoRA term comes from the GEMM) reads as -1, like a position past the unit.
template <int NTOK, typename F>
__device__ __forceinline__ void gather_issue(const LoraLaunch& L, const lora_segments& seg, const Unit& U, int lane,
                                             F tok_index, Gathered& G) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int j = lane + 32 * h;
    G.pa[h] = j < U.r ? __ldg(U.tab + j) : -1;
    G.pb[h] = j < U.r ? __ldg(U.tab + LORA_MAX_RANK + j) : -1;
  }
#pragma unroll
  for (int k = 0; k < NTOK; ++k) {
    const int t = tok_index(lane, k);
    G.tok[k] = t < U.n_tok ? __ldg(seg.perm + U.t_begin + t) : -1;
  }
  if (L.tile_plan != nullptr && U.mixed) {
#pragma unroll
    for (int k = 0; k < NTOK; ++k)
      if (G.tok[k] >= 0 && __ldg(L.tile_plan + (size_t)(G.tok[k] / kTileTokens) * kPlanStride) >= 0) G.tok[k] = -1;
  }
}
__device__ __forceinline__ bool page_ok(int32_t p, int64_t num_pages) { return p >= 0 && p < num_pages; }
// Bit j set when rank column j < r has both pages inside the pool (same value in every lane).
__device__ __forceinline__ uint64_t valid_mask(const Gathered& G, int r, int64_t num_pages, int lane) {
  uint64_t m = 0;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const bool ok = lane + 32 * h < r && page_ok(G.pa[h], num_pages) && page_ok(G.pb[h], num_pages);
    m |= (uint64_t)__ballot_sync(0xffffffffu, ok) << (32 * h);
  }
  return m;
}
__device__ __forceinline__ bool slot_has_lora(const Gathered& G) {
  return __shfl_sync(0xffffffffu, G.pa[0], 0) >= 0;    // page table entry 0 of the slot
}
__device__ __forceinline__ void st_async_v4(uint32_t local_addr, uint32_t local_bar, uint32_t rank, const float (&v)[4]) {
  uint32_t ra, rb;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(local_addr), "r"(rank));
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(rb) : "r"(local_bar), "r"(rank));
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(ra),
               "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "r"(rb)
               : "memory");
}

// FBW: features per block (1024, or 1280 for a 1280-feature share).  Nine warps put three on one
// SM sub-partition, which caps a thread at 168 registers.
template <int KC, int FBW>
__global__ void __launch_bounds__(kThreads, 1)
lora_delta_kernel(LoraLaunch L, lora_segments seg) {
  constexpr int kCluster = KC;                            // CTAs per item, one feature share each
  using R = Ring<FBW>;
  constexpr int kFB = FBW, kRows = R::kRows, kStages = R::kStages, kGps = R::kGroups, kMT = R::kMT;
  constexpr int kRowBytes = R::kRowBytes, kSlotBytes = R::kSlotBytes, kOffX = R::kOffX;
  using SM = Smem<KC>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t q = cluster_rank();
  const uint32_t ring = smem_u32(smem + kOffRing);
  float* part = reinterpret_cast<float*>(smem + kOffPart);
  float* exch = reinterpret_cast<float*>(smem + SM::kOffExch);
  __nv_bfloat16* sb = reinterpret_cast<__nv_bfloat16*>(smem + SM::kOffSb);
  const uint32_t bar_full = smem_u32(smem + SM::kOffBar);
  const uint32_t bar_empty = bar_full + 8 * kMaxStages;
  const uint32_t bar_exch = bar_empty + 8 * kMaxStages;
  const uint32_t bar_xfull = bar_exch + 16, bar_xempty = bar_xfull + 8;
  const uint32_t xbuf = smem_u32(smem + kOffX);

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, kConsumerWarps);
    }
    for (int b = 0; b < 2; ++b) mbar_init(bar_exch + 8 * b, 1);
    mbar_init(bar_xfull, 1);
    mbar_init(bar_xempty, kConsumerWarps);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  cluster_sync_all();                                     // peers' barriers exist before any remote access
  pdl_wait_then_release();

  const int H = L.H;
  const int Hq = H / kCluster;                            // features per CTA (multiple of 16)
  const int n_fb = (Hq + kFB - 1) / kFB;
  const int f_cta = (int)q * Hq;
  const int n_units = *L.n_units;
  const int ng = L.n_group;
  const int n_items = n_units * ng;                       // item i: unit i / ng on member i % ng
  const int n_groups = gridDim.x / kCluster;
  const int group = blockIdx.x / kCluster;
  // Items are dealt to the clusters in waves of n_groups, alternately left to right and right
  // to left.  Units come largest ranks first, so a cluster that draws one of the longest items
  // of a wave draws one of the shortest of the next.  item_at grows with w.
  auto item_at = [n_groups, group](int w) { return w * n_groups + ((w & 1) ? n_groups - 1 - group : group); };

  if (warp == kConsumerWarps) {
    // ================================ producer warp ================================
    // Unit records and page ids are loaded one unit ahead, so their latency hides behind the
    // copies of the current unit.
    auto tok_lane = [](int l, int) { return l; };
    uint32_t it = 0, xi = 0;                              // ring stages and x buffer fills issued
    bool ok = true;
    int4 rec = load_rec(L, item_at(0) / ng, n_units);
    Gathered G;
    Unit U = unit_of(L, rec, item_at(0) % ng);
    gather_issue<1>(L, seg, U, lane, tok_lane, G);
    int4 rec_next = load_rec(L, item_at(1) / ng, n_units);
    for (int w = 0; item_at(w) < n_items && ok; ++w) {   // the producer alone may stop early
      const Unit Un = unit_of(L, rec_next, item_at(w + 1) % ng);
      Gathered Gn;
      gather_issue<1>(L, seg, Un, lane, tok_lane, Gn);
      rec_next = load_rec(L, item_at(w + 2) / ng, n_units);
      if (slot_has_lora(G)) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if (lane + 32 * h < U.r && !(page_ok(G.pa[h], L.num_pages) && page_ok(G.pb[h], L.num_pages))) {
            flag_error(L.err, LORA_DEV_BAD_PAGE);
            G.pa[h] = G.pb[h] = -1;                       // the column is dropped on both sides
          }
        }
        const int nq = (U.r + kRows - 1) / kRows;         // stages of up to kRows rank columns
        // in consumption order: per feature block, the x rows (own buffer) then the A stages;
        // then the B stages.  Lane l < kRows copies rank column kRows q + l of stage q.
        for (int phase = 0; phase < 2 && ok; ++phase) {
          for (int fb = 0; fb < n_fb && ok; ++fb) {
            const int fw = min(kFB, Hq - fb * kFB);
            const int f0 = f_cta + fb * kFB;
            if (phase == 0) {                              // x rows of the unit's tokens
              ok = __all_sync(0xffffffffu, mbar_wait(bar_xempty, (xi & 1) ^ 1));
              if (!ok) break;
              const bool mine = lane < U.n_tok && G.tok[0] >= 0;
              const uint32_t rows = __popc(__ballot_sync(0xffffffffu, mine));
              if (lane == 0) mbar_arrive_expect_tx(bar_xfull, rows * fw * 2);
              __syncwarp();
              if (mine) bulk_g2s(xbuf + lane * kRowBytes, L.x + (int64_t)G.tok[0] * H + f0, fw * 2, bar_xfull);
              ++xi;
            }
            for (int q = 0; q < nq; ++q) {
              const int s = it % kStages;
              ok = __all_sync(0xffffffffu, mbar_wait(bar_empty + 8 * s, ((it / kStages) & 1) ^ 1));
              if (!ok) break;
              // rank column j = kRows q + l is held by lane j % 32 in its entry j / 32 (the lane itself
              // when a stage is 32 columns)
              const int j0 = kRows * q;
              const int32_t held = (j0 >> 5) ? (phase == 0 ? G.pa[1] : G.pb[1]) : (phase == 0 ? G.pa[0] : G.pb[0]);
              const int32_t page = kRows == 32 ? held : __shfl_sync(0xffffffffu, held, (j0 + lane) & 31);
              const bool mine = lane < kRows && page >= 0;
              const uint32_t rows = __popc(__ballot_sync(0xffffffffu, mine));
              if (lane == 0) mbar_arrive_expect_tx(bar_full + 8 * s, rows * fw * 2);
              __syncwarp();
              if (mine) bulk_g2s(ring + s * kSlotBytes + lane * kRowBytes, L.pool + (int64_t)page * H + f0, fw * 2,
                                 bar_full + 8 * s);
              ++it;
            }
          }
        }
      }
      U = Un;
      G = Gn;
    }
    if (!ok) flag_error(L.err, LORA_DEV_WAIT_TIMEOUT);
    // Drain: the most recent use of every slot and of the x buffer has landed before exit.
    if (lane == 0) {
      for (uint32_t k = it > (uint32_t)kStages ? it - kStages : 0; k < it; ++k)
        if (!mbar_wait(bar_full + 8 * (k % kStages), (k / kStages) & 1)) flag_error(L.err, LORA_DEV_WAIT_TIMEOUT);
      if (xi > 0 && !mbar_wait(bar_xfull, (xi - 1) & 1)) flag_error(L.err, LORA_DEV_WAIT_TIMEOUT);
    }
  } else {
    // ================================ consumer warps ================================
    // After a failed wait the warps keep walking the same sequence of units, stages and barriers
    // (skipping the waits), so every named and cluster barrier still sees all its threads.
    // Lane l stores delta for tokens tok_store(l, k), k < 4 (the MMA accumulator layout).
    auto tok_store = [](int l, int k) { return (k >> 1) * 8 + 2 * (l & 3) + (k & 1); };
    uint32_t it = 0, n_done = 0, xi = 0;
    bool ok = true;
    const int mi = lane >> 3, ri = lane & 7;              // ldmatrix: matrix and row this lane addresses
    __nv_bfloat16* sb_hi = sb;
    __nv_bfloat16* sb_lo = sb + kUnitTok * kSbPitch;
    int4 rec = load_rec(L, item_at(0) / ng, n_units);
    Gathered G;
    Unit U = unit_of(L, rec, item_at(0) % ng);
    gather_issue<4>(L, seg, U, lane, tok_store, G);
    int4 rec_next = load_rec(L, item_at(1) / ng, n_units);
    for (int w = 0; item_at(w) < n_items; ++w) {
      const Unit Un = unit_of(L, rec_next, item_at(w + 1) % ng);
      Gathered Gn;
      gather_issue<4>(L, seg, Un, lane, tok_store, Gn);
      rec_next = load_rec(L, item_at(w + 2) / ng, n_units);
      if (slot_has_lora(G)) {
        const uint64_t vm = valid_mask(G, U.r, L.num_pages, lane);
        const int ng = (U.r + 15) / 16;
        const int wpg = kConsumerWarps / ng;              // warps per page group in the shrink
        const int my_g = warp / wpg, sub = warp % wpg;

        // ---- shrink over this CTA's feature share: acc[n-tile] = A_g^T x^T (16 pages x 8 tokens)
        float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        const int nq = (U.r + kRows - 1) / kRows;
        for (int fb = 0; fb < n_fb; ++fb) {
          const int fw = min(kFB, Hq - fb * kFB);
          ok = ok && wait_warp(bar_xfull, xi & 1);
          ++xi;
          for (int q = 0; q < nq; ++q) {
            const int s = it % kStages;
            ok = ok && wait_warp(bar_full + 8 * s, (it / kStages) & 1);
            ++it;
            if (ok && my_g / kGps == q && my_g < ng) {   // this warp's group: rows 16 (my_g % kGps) ..
              const uint32_t abase = ring + s * kSlotBytes + (my_g % kGps) * 16 * kRowBytes;
              const uint32_t a_row = abase + (ri + 8 * (mi & 1)) * kRowBytes + 16 * (mi >> 1);
              const uint32_t x_row = xbuf + (ri + 8 * (mi >> 1)) * kRowBytes + 16 * (mi & 1);
#pragma unroll 4
              for (int ks = sub; ks < fw / 16; ks += wpg) {
                uint32_t af[4], xf[4];
                ldsm_x4(a_row + ks * 32, af);
                ldsm_x4(x_row + ks * 32, xf);
                mma_bf16(acc[0], af, xf[0], xf[1]);
                mma_bf16(acc[1], af, xf[2], xf[3]);
              }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_empty + 8 * s);
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_xempty);            // the x rows may be replaced
        }
        // partial sums of this warp: part[warp][page][token]
        if (my_g < ng) {
          float* pw = part + warp * 256;
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) {
            const int m = lane >> 2, n = nt * 8 + 2 * (lane & 3);
            pw[m * 16 + n] = acc[nt][0];
            pw[m * 16 + n + 1] = acc[nt][1];
            pw[(m + 8) * 16 + n] = acc[nt][2];
            pw[(m + 8) * 16 + n + 1] = acc[nt][3];
          }
        }
        consumer_sync();
        // This CTA's partial of s over its share goes to all KC CTAs, exch[b][q][j][t], as
        // asynchronous remote stores that count their bytes on the receiver's barrier.
        const int b = n_done & 1;
        if (tid == 0) mbar_arrive_expect_tx(bar_exch + 8 * b, kCluster * ng * 256 * 4);
        if (tid < ng * 64) {
          const int j = tid >> 2, t0 = (tid & 3) * 4, g = j >> 4;
          float v[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            float acc_v = 0.f;
            for (int k = 0; k < wpg; ++k) acc_v += part[(g * wpg + k) * 256 + (j & 15) * 16 + t0 + i];
            v[i] = (((vm >> j) & 1) && t0 + i < U.n_tok) ? acc_v : 0.f;
          }
          const uint32_t dst = smem_u32(exch + ((b * kCluster + q) * LORA_MAX_RANK + j) * kUnitTok + t0);
#pragma unroll
          for (int c = 0; c < kCluster; ++c) st_async_v4(dst, bar_exch + 8 * b, (uint32_t)c, v);
        }
        ok = ok && wait_warp(bar_exch + 8 * b, (n_done >> 1) & 1);
        ++n_done;
        // s = sum of the KC shares in cluster-rank order, split into bf16 hi + lo, token-major
        for (int e = tid; e < ng * 256; e += kConsumers) {
          const int j = e >> 4, t = e & 15;
          const float* ex = exch + (b * kCluster * LORA_MAX_RANK + j) * kUnitTok + t;
          float v = ex[0];
#pragma unroll
          for (int c = 1; c < kCluster; ++c) v += ex[c * LORA_MAX_RANK * kUnitTok];
          const __nv_bfloat16 hi = __float2bfloat16_rn(v);
          sb_hi[t * kSbPitch + j] = hi;
          sb_lo[t * kSbPitch + j] = __float2bfloat16_rn(v - __bfloat162float(hi));
        }
        consumer_sync();

        // ---- expand: delta[t][f] for this CTA's features, warp w owns 16 kMT features per block
        for (int fb = 0; fb < n_fb; ++fb) {
          const int fw = min(kFB, Hq - fb * kFB);
          const int f_warp = warp * 16 * kMT;
          float e[kMT][2][4];
#pragma unroll
          for (int mt = 0; mt < kMT; ++mt)
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
              for (int k = 0; k < 4; ++k) e[mt][nt][k] = 0.f;
          for (int q = 0; q < nq; ++q) {
            const int s = it % kStages;
            ok = ok && wait_warp(bar_full + 8 * s, (it / kStages) & 1);
            ++it;
            for (int g = kGps * q; g < min(ng, kGps * q + kGps) && ok && f_warp < fw; ++g) {
              uint32_t sh[4], sl[4];
              const uint32_t s_off = ((ri + 8 * (mi >> 1)) * kSbPitch + 16 * g + 8 * (mi & 1)) * 2;
              ldsm_x4(smem_u32(sb_hi) + s_off, sh);
              ldsm_x4(smem_u32(sb_lo) + s_off, sl);
              // A-fragment elements of page columns without valid pages are zeroed
              const uint32_t kb = 16 * g + 2 * (lane & 3);
              const uint32_t m01 = (((vm >> kb) & 1) ? 0x0000FFFFu : 0u) | (((vm >> (kb + 1)) & 1) ? 0xFFFF0000u : 0u);
              const uint32_t m23 = (((vm >> (kb + 8)) & 1) ? 0x0000FFFFu : 0u) | (((vm >> (kb + 9)) & 1) ? 0xFFFF0000u : 0u);
              const uint32_t b_row =
                  ring + s * kSlotBytes + ((g % kGps) * 16 + ri + 8 * (mi >> 1)) * kRowBytes + 16 * (mi & 1);
#pragma unroll
              for (int mt = 0; mt < kMT; ++mt) {
                if (f_warp + mt * 16 < fw) {
                  uint32_t af[4];
                  ldsm_x4_t(b_row + (f_warp + mt * 16) * 2, af);
                  af[0] &= m01;
                  af[1] &= m01;
                  af[2] &= m23;
                  af[3] &= m23;
                  mma_bf16(e[mt][0], af, sh[0], sh[1]);
                  mma_bf16(e[mt][0], af, sl[0], sl[1]);
                  mma_bf16(e[mt][1], af, sh[2], sh[3]);
                  mma_bf16(e[mt][1], af, sl[2], sl[3]);
                }
              }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_empty + 8 * s);
          }
          if (!ok) continue;
          // store the valid tokens' rows of delta
          const int fbase = f_cta + fb * kFB + f_warp + (lane >> 2);
#pragma unroll
          for (int mt = 0; mt < kMT; ++mt) {
            if (f_warp + mt * 16 < fw) {
#pragma unroll
              for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                  const int tk = G.tok[nt * 2 + (k & 1)];
                  if (tk >= 0) U.delta[(int64_t)tk * H + fbase + mt * 16 + 8 * (k >> 1)] = e[mt][nt][k];
                }
            }
          }
        }
      }
      U = Un;
      G = Gn;
    }
    if (!ok && lane == 0) flag_error(L.err, LORA_DEV_WAIT_TIMEOUT);
  }
  cluster_sync_all();                                     // no CTA leaves while a peer may still address it
}

template <int KC, int FBW>
int active_clusters() {
  static int cached[kMaxDeviceFlags] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  const bool cache = dev >= 0 && dev < kMaxDeviceFlags;
  if (cache && cached[dev] > 0) return cached[dev];
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(KC * 64);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Smem<KC>::kBytes;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = KC;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, lora_delta_kernel<KC, FBW>, &cfg) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    n = device_sm_count() / KC;
  }
  if (cache) cached[dev] = n;
  return n;
}

template <int KC, int FBW>
int launch_delta_kc(const LoraLaunch& L, cudaStream_t st) {
  static DeviceFlags attr;
  int rc = ensure_smem_attr(attr, lora_delta_kernel<KC, FBW>, Smem<KC>::kBytes,
                            "lora_delta_kernel: shared memory attribute");
  if (rc != LORA_OK) return rc;
  // Persistent clusters, as many as can be resident; each loops over the units.
  int groups = active_clusters<KC, FBW>();
  const int item_cap = L.seg->unit_cap * L.n_group;
  if (item_cap < groups) groups = item_cap > 0 ? item_cap : 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(groups * KC);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Smem<KC>::kBytes;
  cfg.stream = st;
  cudaLaunchAttribute attrs[2];
  attrs[0].id = cudaLaunchAttributeClusterDimension;
  attrs[0].val.clusterDim.x = KC;
  attrs[0].val.clusterDim.y = 1;
  attrs[0].val.clusterDim.z = 1;
  attrs[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = L.pdl ? 2 : 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, lora_delta_kernel<KC, FBW>, L, *L.seg);
  if (e == cudaSuccess) e = cudaGetLastError();
  return e == cudaSuccess ? LORA_OK : lora_cuda_fail(e, "lora_delta_kernel launch");
}

}  // namespace

// The feature split of an item: 2 CTAs when their halves are at most 1024 features (H <= 2048:
// twice as many items run at once), else 4.  A split into 5 made the kernel alone faster but a
// layer's chain of kernels slower: its 150 SMs leave no room for the next kernel to start early.
int delta_split(int32_t H) { return H <= 2048 ? 2 : 4; }

// Feature blocks of 1024, except a CTA share of 1025..1280 features, which is one block.
int launch_lora_delta(const LoraLaunch& L, cudaStream_t st) {
  if (delta_split(L.H) == 2) return launch_delta_kc<2, 1024>(L, st);
  const int Hq = L.H / 4;
  return Hq > 1024 && Hq <= 1280 ? launch_delta_kc<4, 1280>(L, st) : launch_delta_kc<4, 1024>(L, st);
}
