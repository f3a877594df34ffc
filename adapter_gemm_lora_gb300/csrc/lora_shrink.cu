// Shrink of the fused tiles of a prefill-shaped batch: s = x A for every token of a 256-token tile
// that carries at most LORA_TILE_ADAPTERS adapters, written as bf16 hi and lo parts for the base
// GEMM, which then adds (x A) B inside its own accumulator.
//
// "S-LoRA, in depth", section "Merge or keep adapters separate": the unmerged term is (xA)B;
// section "Kernels for a batch of mixed ranks": when many tokens share an adapter (prefill), the
// shrink is a small matrix product per adapter over its pages.  Here it runs on the tensor cores:
// in swap-AB form (as the base GEMM), M = the adapter's A pages (64 rows per slot, two slots per
// tile of 128 rows), N = the 256 tokens of the tile, K = H.
//
// Work item: one fused (tile, adapter slot b) entry of the segment plan, for a pair of slots of
// the call's group (rows 0..63: slot 2p, rows 64..127: slot 2p+1).  A cluster of 4 CTAs takes an
// item, CTA q streaming the K quarter [q H/4, (q+1) H/4): warp 0 loads the tile's x rows with TMA,
// warps 2-5 gather the A page rows of the quarter with 16-byte cp.async copies straight into the
// 128-byte-swizzled K-major layout the MMA reads (a page row is 64 K values per stage: 128 B, the
// swizzle atom's row), warp 1 issues the tcgen05 MMAs into one of two TMEM accumulators, and
// warps 6-9 finish the previous item meanwhile.  Finishing: CTA q owns tokens [64q, 64q + 64) of
// the tile; every CTA writes its partial sums of the other owners' tokens to a scratch block in
// global memory (L2) and signals each owner on an mbarrier in the owner's shared memory (remote
// arrive, cluster-scope release); the owner adds the four partials in rank order, the same order
// for every token, and writes its tokens' rows of s.  A token's row gets s in the columns of
// tile slot b only when the token's adapter is the entry's adapter; every other token of the tile
// gets zeros there, so the GEMM may multiply the whole tile by the entry's B pages.
//
// Precision: bf16 products, fp32 accumulation in TMEM and in the rank-order sum; s is split into
// hi = bf16(s) and lo = bf16(s - hi) (16 bits of mantissa), as in the gather kernel.
// Every wait is bounded (~2 s); a CTA that gives up raises the device error word and stops.
#include "tc_ptx.h"

namespace {

constexpr int BM = 128;                      // A rows per item (two slots of 64)
constexpr int BN = kTileTokens;              // tokens per tile
constexpr int BK = 64;
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;         // 16 KB
constexpr int X_BYTES = BN * BK * 2;         // 32 KB
constexpr int STAGE_BYTES = A_BYTES + X_BYTES;
constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + 256;
constexpr int KS = kShrinkCluster;           // CTAs per item, one K quarter each
constexpr int THREADS = 320;                 // TMA, MMA, 4 loader warps, 4 finishing warps
constexpr int LOADERS = 128;
constexpr int OWN = BN / KS;                 // tokens each CTA finishes (64)
constexpr size_t BLOCK_FLOATS = (size_t)OWN * BM;                   // one partial block
constexpr size_t REGION_FLOATS = (size_t)KS * (KS - 1) * BLOCK_FLOATS;  // one item's exchange
static_assert(kShrinkScratchFloats >= (size_t)kShrinkMaxClusters * 2 * REGION_FLOATS,
              "exchange scratch: two regions (item parity) per cluster");

struct ShrinkParams {
  const uint16_t* pool;
  int64_t num_pages;
  int32_t H, T, n_slots, n_group, n_kb;
  int32_t slot[LORA_MAX_GROUP];
  uint16_t* s_out[LORA_MAX_GROUP];           // [T_max][kSCols] bf16 per group member
  const int32_t* ptab;
  const int32_t* rank;
  const int32_t* tile_plan;
  const int32_t* entries;
  const int32_t* n_entries;
  const int32_t* tok_adapter;
  float* scratch;
  int32_t* err;
};

struct Item {
  int tile, b, a, r, pair;
};
__device__ __forceinline__ Item item_of(const ShrinkParams& p, int i, int n_pairs) {
  Item it;
  const int e = __ldg(p.entries + i / n_pairs);
  it.tile = e / kTileAdapters;
  it.b = e % kTileAdapters;
  it.a = __ldg(p.tile_plan + (size_t)it.tile * kPlanStride + 1 + it.b);
  it.r = it.a >= 0 ? __ldg(p.rank + it.a) : 0;
  if (it.r < 0 || it.r > LORA_MAX_RANK) it.r = 0;
  it.pair = i % n_pairs;
  return it;
}
// Page-table row of A pages of adapter a on group member g (nullptr: no such member, or no LoRA
// on that slot).
__device__ __forceinline__ const int32_t* a_pages(const ShrinkParams& p, const Item& it, int g) {
  if (g >= p.n_group || it.a < 0) return nullptr;
  int slot = p.slot[0];
#pragma unroll
  for (int k = 1; k < LORA_MAX_GROUP; ++k)
    if (g == k) slot = p.slot[k];
  const int32_t* tab = p.ptab + ((int64_t)it.a * p.n_slots + slot) * kTabStride;
  return __ldg(tab) >= 0 ? tab : nullptr;
}

__global__ void __launch_bounds__(THREADS, 1)
lora_shrink_kernel(const __grid_constant__ CUtensorMap tm_x, ShrinkParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t s_base = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
  const uint32_t bar_full = smem_u32(bars);                 // [STAGES] x rows landed (TMA)
  const uint32_t bar_afull = bar_full + 8 * STAGES;          // [STAGES] A rows landed (4 loader warps)
  const uint32_t bar_empty = bar_afull + 8 * STAGES;         // [STAGES] stage consumed (MMA commit)
  const uint32_t bar_tfull = bar_empty + 8 * STAGES;         // [2] accumulator complete
  const uint32_t bar_tempty = bar_tfull + 16;                // [2] accumulator drained (4 warps)
  const uint32_t bar_ready = bar_tempty + 16;                // [2] peers' partials written (12 warps)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 3 * STAGES + 6);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int me = (int)cluster_ctarank();
  const int n_clusters = (int)gridDim.x / KS;
  const int cluster_id = (int)blockIdx.x / KS;
  const int kb_lo = me * p.n_kb / KS, kb_hi = (me + 1) * p.n_kb / KS;
  const int nk = kb_hi - kb_lo;                              // >= 1: the launcher requires n_kb >= 4
  pdl_wait_then_release();                                   // the plan comes from the segment build
  const int n_pairs = (p.n_group + 1) / 2;
  const int n_items = *p.n_entries * n_pairs;
  if (cluster_id >= n_items) return;                         // the whole cluster: nothing to do

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_afull + 8 * s, LOADERS / 32);
      mbar_init(bar_empty + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_tfull + 8 * b, 1);
      mbar_init(bar_tempty + 8 * b, 4);
      mbar_init(bar_ready + 8 * b, (KS - 1) * 4);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_x)) : "memory");
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 2 * BN);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync_all();                                        // peers' barriers exist before any remote arrive
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {                                         // TMA: the tile's x rows, K quarter
      const uint64_t pol = policy_evict_last();              // read again by the other items of the tile
      uint32_t it = 0;
      bool ok = true;
      for (int i = cluster_id; i < n_items && ok; i += n_clusters) {
        const Item item = item_of(p, i, n_pairs);
        for (int k = 0; k < nk; ++k, ++it) {
          const int s = it % STAGES;
          if (!mbar_wait(bar_empty + 8 * s, ((it / STAGES) & 1) ^ 1)) {
            flag_error(p.err, LORA_DEV_WAIT_TIMEOUT);
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(bar_full + 8 * s, X_BYTES);
          tma_load_2d(s_base + s * STAGE_BYTES + A_BYTES, &tm_x, (kb_lo + k) * BK, item.tile * BN, bar_full + 8 * s, pol);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {                                         // MMA issuer
      const uint32_t idesc = make_idesc_bf16(BM, BN);
      uint32_t it = 0;
      int n = 0;
      bool ok = true;
      for (int i = cluster_id; i < n_items && ok; i += n_clusters, ++n) {
        const int b = n & 1;
        if (!mbar_wait(bar_tempty + 8 * b, ((n >> 1) & 1) ^ 1)) {
          flag_error(p.err, LORA_DEV_WAIT_TIMEOUT);
          break;
        }
        tc_fence_after();
        const uint32_t acc = tmem + (uint32_t)(b * BN);
        for (int k = 0; k < nk; ++k, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1;
          if (!mbar_wait(bar_full + 8 * s, ph) || !mbar_wait(bar_afull + 8 * s, ph)) {
            flag_error(p.err, LORA_DEV_WAIT_TIMEOUT);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = s_base + s * STAGE_BYTES;
          const uint64_t ad = sw128_kmajor_desc(st);
          const uint64_t bd = sw128_kmajor_desc(st + A_BYTES);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) mma_bf16_ss(acc, ad + 2 * kk, bd + 2 * kk, idesc, (k | kk) != 0);
          mma_commit(bar_empty + 8 * s);
        }
        if (ok) mma_commit(bar_tfull + 8 * b);
      }
    }
    __syncwarp();
  } else if (warp < 6) {
    // ---- loaders: thread l copies 16-byte chunk (l & 7) of A rows (l >> 3) + 16 i, i < 8 ----
    const int l = threadIdx.x - 64;
    const int ch = l & 7;
    uint32_t it = 0;
    bool ok = true;
    for (int i = cluster_id; i < n_items && ok; i += n_clusters) {
      const Item item = item_of(p, i, n_pairs);
      const int32_t* tab0 = a_pages(p, item, 2 * item.pair);
      const int32_t* tab1 = a_pages(p, item, 2 * item.pair + 1);
      int64_t page[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int row = (l >> 3) + 16 * q;
        const int j = row & 63;
        const int32_t* tab = (row >> 6) ? tab1 : tab0;
        page[q] = -1;                                          // row not copied: its sums are never read
        if (tab != nullptr && j < item.r) {
          const int32_t pg = __ldg(tab + j);
          if (pg >= 0 && pg < p.num_pages) {
            page[q] = pg;
          } else {
            flag_error(p.err, LORA_DEV_BAD_PAGE);
            page[q] = -2;                                      // zero row: the column is dropped
          }
        }
      }
      for (int k = 0; k < nk; ++k, ++it) {
        const int s = it % STAGES;
        ok = __all_sync(0xffffffffu, mbar_wait(bar_empty + 8 * s, ((it / STAGES) & 1) ^ 1));
        if (!ok) break;
        const uint32_t st = s_base + s * STAGE_BYTES;
        const int k0 = (kb_lo + k) * BK + ch * 8;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const int row = (l >> 3) + 16 * q;
          if (page[q] != -1)
            cp_async_16(st + (uint32_t)(row >> 3) * 1024u + sw128_offset(row, ch),
                        p.pool + (page[q] >= 0 ? page[q] * p.H + k0 : 0), page[q] >= 0);
        }
        cp_async_commit();
        if (k >= 2) {                                          // the copies of stage it - 2 have landed
          cp_async_wait<2>();
          fence_proxy_async_shared();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_afull + 8 * ((it - 2) % STAGES));
        }
      }
      // the item's last stages
      cp_async_wait<0>();
      fence_proxy_async_shared();
      __syncwarp();
      if (ok && lane == 0)
        for (int k = nk < 2 ? 0 : nk - 2; k < nk; ++k) mbar_arrive(bar_afull + 8 * ((it - nk + k) % STAGES));
    }
    if (!ok && lane == 0) flag_error(p.err, LORA_DEV_WAIT_TIMEOUT);
  } else {
    // ---- finishing warps: TMEM lane quarter (warp & 3) = A rows 32 (warp & 3) .. + 31 ----
    const int qw = warp & 3;
    const int row = qw * 32 + lane;
    const int h = row >> 6, j = row & 63;
    int n = 0;
    for (int i = cluster_id; i < n_items; i += n_clusters, ++n) {
      const Item item = item_of(p, i, n_pairs);
      const int b = n & 1;
      const uint32_t ph = (n >> 1) & 1;
      const int g = 2 * item.pair + h;
      const bool valid_row = j < item.r && a_pages(p, item, g) != nullptr;
      uint16_t* s_out = p.s_out[0];
#pragma unroll
      for (int k = 1; k < LORA_MAX_GROUP; ++k)
        if (g == k) s_out = p.s_out[k];
      bool ok = __all_sync(0xffffffffu, mbar_wait(bar_tfull + 8 * b, ph));
      if (!ok) {
        if (lane == 0) flag_error(p.err, LORA_DEV_WAIT_TIMEOUT);
        break;
      }
      tc_fence_after();
      const uint32_t acc_row = tmem + (uint32_t)(b * BN) + ((uint32_t)(qw * 32) << 16);
      float* region = p.scratch + (size_t)(cluster_id * 2 + (n & 1)) * REGION_FLOATS;
      // 1. partial sums of the other owners' tokens: block (owner o, sender me) is [64 tokens][128 rows]
      for (int o = 0; o < KS; ++o) {
        if (o == me) continue;
        float* dst = region + (size_t)(o * (KS - 1) + (me < o ? me : me - 1)) * BLOCK_FLOATS + row;
#pragma unroll 1
        for (int c = 0; c < OWN; c += 16) {
          uint32_t v[16];
          tmem_ld_32x32b_x16(acc_row + (uint32_t)(o * OWN + c), v);
          tmem_ld_wait();
#pragma unroll
          for (int t = 0; t < 16; ++t) dst[(size_t)(c + t) * BM] = __uint_as_float(v[t]);
        }
      }
      __syncwarp();
      if (lane == 0) {
        asm volatile("fence.acq_rel.cluster;" ::: "memory");
#pragma unroll
        for (int o = 0; o < KS; ++o)
          if (o != me) mbar_arrive_remote_release(bar_ready + 8 * b, (uint32_t)o);
      }
      __syncwarp();
      // 2. own tokens: the four partials in rank order, then the rows of s
      ok = __all_sync(0xffffffffu, mbar_wait_acq_cluster(bar_ready + 8 * b, ph));
      if (!ok) {
        if (lane == 0) flag_error(p.err, LORA_DEV_WAIT_TIMEOUT);
        break;
      }
      const float* in0 = region + (size_t)(me * (KS - 1)) * BLOCK_FLOATS + row;
#pragma unroll 1
      for (int c = 0; c < OWN; c += 16) {
        const int t0 = item.tile * BN + me * OWN + c;
        int32_t ta[16];
#pragma unroll
        for (int t = 0; t < 16; ++t) ta[t] = t0 + t < p.T ? __ldg(p.tok_adapter + t0 + t) : -1;
        uint32_t v[16];
        tmem_ld_32x32b_x16(acc_row + (uint32_t)(me * OWN + c), v);
        tmem_ld_wait();
        float pv[KS - 1][16];
#pragma unroll
        for (int q = 0; q < KS - 1; ++q)
#pragma unroll
          for (int t = 0; t < 16; ++t) pv[q][t] = __ldcg(in0 + (size_t)q * BLOCK_FLOATS + (size_t)(c + t) * BM);
        if (g < p.n_group) {
#pragma unroll
          for (int t = 0; t < 16; ++t) {
            float sum = me == 0 ? __uint_as_float(v[t]) : pv[0][t];
#pragma unroll
            for (int src = 1; src < KS; ++src) {
              const float peer = src < me ? pv[src < KS - 1 ? src : KS - 2][t] : pv[src - 1][t];
              sum += src == me ? __uint_as_float(v[t]) : peer;
            }
            if (t0 + t < p.T) {
              const float sv = (valid_row && ta[t] == item.a) ? sum : 0.f;
              const __nv_bfloat16 hi = __float2bfloat16_rn(sv);
              const __nv_bfloat16 lo = __float2bfloat16_rn(sv - __bfloat162float(hi));
              uint16_t* dst = s_out + (size_t)(t0 + t) * kSCols + item.b * 2 * LORA_MAX_RANK + j;
              dst[0] = __bfloat16_as_ushort(hi);
              dst[LORA_MAX_RANK] = __bfloat16_as_ushort(lo);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_tempty + 8 * b);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, 2 * BN);
  cluster_sync_all();                                        // no peer may still arrive on this CTA's barriers
}

int shrink_clusters() {
  static int cached[kMaxDeviceFlags] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  const bool cache = dev >= 0 && dev < kMaxDeviceFlags;
  if (cache && cached[dev] > 0) return cached[dev];
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(KS * 64);
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = KS;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, lora_shrink_kernel, &cfg) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    n = device_sm_count() / KS;
  }
  if (n > kShrinkMaxClusters) n = kShrinkMaxClusters;
  if (cache) cached[dev] = n;
  return n;
}

}  // namespace

int launch_lora_shrink(const ShrinkLaunch& S, cudaStream_t st) {
  static DeviceFlags attr;
  int rc = ensure_smem_attr(attr, lora_shrink_kernel, SMEM_BYTES, "lora_shrink_kernel: shared memory attribute");
  if (rc != LORA_OK) return rc;
  const lora_segments* seg = S.seg;
  if (S.H / BK < KS || S.n_group < 1 || S.n_group > LORA_MAX_GROUP || !seg->s_lora || !seg->shrink_scratch)
    return lora_fail(LORA_EINVAL, "lora_shrink: batch or workspace without fused tiles");
  CUtensorMap tm_x;
  rc = encode_2d(&tm_x, S.x, (uint64_t)S.H, (uint64_t)S.T, (uint32_t)BN);
  if (rc != LORA_OK) return rc;
  ShrinkParams P = {};
  P.pool = S.pool;
  P.num_pages = S.num_pages;
  P.H = S.H;
  P.T = S.T;
  P.n_slots = S.n_slots;
  P.n_group = S.n_group;
  P.n_kb = S.H / BK;
  for (int i = 0; i < LORA_MAX_GROUP; ++i) {
    const int k = i < S.n_group ? i : 0;
    P.slot[i] = S.slot[k];
    P.s_out[i] = seg->s_lora + (size_t)k * seg->T_max * kSCols;
  }
  P.ptab = S.ptab;
  P.rank = S.rank;
  P.tile_plan = seg->tile_plan;
  P.entries = seg->entries;
  P.n_entries = seg->n_entries;
  P.tok_adapter = seg->tok_adapter;
  P.scratch = seg->shrink_scratch;
  P.err = S.err;
  int clusters = shrink_clusters();
  const int items_max = ((S.T + BN - 1) / BN) * kTileAdapters * ((S.n_group + 1) / 2);
  if (clusters > items_max) clusters = items_max;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(clusters * KS);
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = st;
  cudaLaunchAttribute attrs[2];
  attrs[0].id = cudaLaunchAttributeClusterDimension;
  attrs[0].val.clusterDim.x = KS;
  attrs[0].val.clusterDim.y = 1;
  attrs[0].val.clusterDim.z = 1;
  attrs[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = S.pdl ? 2 : 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, lora_shrink_kernel, tm_x, P);
  if (e == cudaSuccess) e = cudaGetLastError();
  return e == cudaSuccess ? LORA_OK : lora_cuda_fail(e, "lora_shrink_kernel launch");
}
