// Base projection x W^T on the 5th-generation tensor cores (tcgen05 + TMEM), fed by TMA,
// with a fused epilogue that adds the LoRA delta before the single rounding to bf16.
//
// "S-LoRA, in depth", section "Merge or keep adapters separate": the expensive xW product
// is batched across every request regardless of adapter; section "The architecture": each
// layer runs the base projection for the whole batch.  This is the only dense contraction
// of the path.
//
// Orientation (swap-AB): the MMA's M side is the output feature n (rows of W[out][in]),
// its N side the token t, K the hidden index.  Both operands are K-major, which is how
// W (nn.Linear layout) and x (row-major tokens) sit in memory, so TMA copies 64-wide
// K-slices of each straight into the 128-byte-swizzled shared-memory layout the MMA
// reads.  The accumulator tile D[n, t] (128 x BN fp32) lives in TMEM: lane = feature,
// column = token.  That suits the epilogue: a warp covers 32 consecutive features of
// one token, so delta loads and y stores are contiguous along the feature dimension.
//
// Per CTA: one 128 x BN output tile over the full K.  Warp 0 issues TMA loads into a ring
// of up to 8 stages (each 1, 2 or 4 K chunks of 64, so that a stage carries >= ~40 KB), warp 1 owns TMEM and a single thread issues the MMAs, then all 8 warps
// drain TMEM (warp w reads TMEM lanes 32*(w%4) .. +31, half the columns each).
// Token tiles shrink (down to 32 tokens) until the grid fills the SMs.  Every CTA loads its own
// W tile; CTAs that share a feature tile meet in L2, which holds W across them.
// The epilogue stages the fp32 delta sub-tile (one TMA load) and the bf16 output (one TMA
// store) through the freed stage memory.  The mainloop reads only x and W, so the kernel is
// launched as a programmatic dependent of the LoRA kernels before it and waits for them
// (griddepcontrol.wait) only before its epilogue reads the delta.
// Every mbarrier wait is bounded (~2 s of SM cycles); on expiry the CTA raises the device error word,
// skips the rest of its work and frees TMEM before returning.
#include "tc_ptx.h"

namespace {

constexpr int BM = 128;          // output features per tile (MMA M)
constexpr int BK = 64;           // K elements per stage: one 128-byte swizzle atom wide
constexpr int MAX_BN = 256;      // tokens per tile (MMA N)
constexpr int MAX_STAGES = 8;
constexpr int A_BYTES = BM * BK * 2;
constexpr int STAGE_AREA = 192 * 1024;        // ring of stages; reused by the epilogue
constexpr int BAR_BYTES = 512;
constexpr int SMEM_BYTES = 1024 + STAGE_AREA + BAR_BYTES;
constexpr int THREADS = 256;

struct GemmParams {
  uint16_t* y;
  const float* delta;
  float* partials;
  const int32_t* tok_adapter;
  const int32_t* ptab;
  int32_t* err;
  int32_t T, H, BN, n_kb, kc, stages, ks, slot, n_slots;
};


// Ballot masks of the tokens (columns) that carry LoRA on this slot, for the 32-column chunks
// c0, c0 + step, ... (at most 4): all id loads are issued before any page-table load, so the two
// dependent global reads cost one latency each for every chunk of the warp together.
__device__ __forceinline__ void presence_masks(const GemmParams& p, int slot, int t_col0, int c0, int step, int c_end,
                                               int lane, unsigned (&pm)[4]) {
  int a[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int c = c0 + k * step;
    const int tl = t_col0 + c * 32 + lane;
    a[k] = (c < c_end && tl < p.T) ? p.tok_adapter[tl] : -1;
  }
  int present[4];
#pragma unroll
  for (int k = 0; k < 4; ++k)
    present[k] = a[k] >= 0 ? p.ptab[((int64_t)a[k] * p.n_slots + slot) * kTabStride] >= 0 : 0;
#pragma unroll
  for (int k = 0; k < 4; ++k) pm[k] = __ballot_sync(0xffffffffu, present[k]);
}


// Epilogue when K is split over a cluster of ks CTAs (one token tile of BN columns).  CTA `me`
// owns token columns [me*w, (me+1)*w), w = BN/ks.  Every CTA writes the fp32 partial sums of
// the other owners' columns from TMEM to a global scratch block (coalesced, stays in L2); after
// a cluster barrier each owner reads the ks-1 blocks of its columns, adds the ks partials in
// cluster-rank order (the same order in every CTA), adds the delta and writes its columns of y
// straight from registers.  Scratch block of (owner o, sender s): [w tokens][128 features] at
// index (m_tile * ks + o) * (ks - 1) + (s < o ? s : s - 1).
template <int KS>
__device__ __forceinline__ void split_k_epilogue(const GemmParams& p, uint32_t tmem_row, int m0, int t0, int me, int row,
                                                 int lane, int h, bool ok) {
  constexpr int ks = KS;
  const int w = p.BN / ks;
  const int m_tile = m0 / BM;
  const int feat = m0 + row;                      // this thread's output feature
  const size_t blk = (size_t)w * BM;
  // The scratch was last read by the GEMM launch before this one, and the delta and ids come
  // from the kernels before this one: wait for them before writing or reading.
  pdl_wait_then_release();
  if (ok) {
    for (int c = h; c < p.BN / 32; c += 2) {      // other owners' columns: this CTA's partials
      const int o = (c * 32) / w;
      if (o == me) continue;
      uint32_t v[32];
      tmem_ld_32x32b_x32(tmem_row + (uint32_t)(c * 32), v);
      tmem_ld_wait();
      float* dst = p.partials + (size_t)((m_tile * ks + o) * (ks - 1) + (me < o ? me : me - 1)) * blk +
                   (size_t)(c * 32 - o * w) * BM + row;
#pragma unroll
      for (int i = 0; i < 32; ++i) dst[(size_t)i * BM] = __uint_as_float(v[i]);
    }
  }
  __threadfence();                                // this thread's partials are visible GPU-wide
  // Loads for the first own chunk go out before the barrier and stay in flight across it: the
  // delta column block (selected by the presence mask later) and the presence lookups.
  const int c_first = me * (w / 32) + h, c_end = (me + 1) * (w / 32);
  float dv[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const int t = t0 + c_first * 32 + i;
    dv[i] = (c_first < c_end && t < p.T && feat < p.H) ? __ldg(p.delta + (size_t)t * p.H + feat) : 0.f;
  }
  unsigned pm[4];                                 // own chunks c_first + 2k
  presence_masks(p, p.slot, t0, c_first, 2, c_end, lane, pm);
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");   // all partials of the cluster
  if (!ok) return;
#pragma unroll 1
  for (int k = 0; k < 4; ++k) {                   // own columns
    const int c = c_first + 2 * k;
    if (c >= c_end) break;
    uint32_t v[32];
    tmem_ld_32x32b_x32(tmem_row + (uint32_t)(c * 32), v);
    tmem_ld_wait();
    const unsigned pmask = k == 0 ? pm[0] : k == 1 ? pm[1] : k == 2 ? pm[2] : pm[3];
    const size_t off0 = (size_t)(c * 32 - me * w) * BM + row;
    const float* in0 = p.partials + (size_t)(m_tile * ks + me) * (ks - 1) * blk + off0;
    const int tc = t0 + c * 32;
    if (k > 0) {
#pragma unroll
      for (int i = 0; i < 32; ++i)
        dv[i] = (tc + i < p.T && feat < p.H) ? __ldg(p.delta + (size_t)(tc + i) * p.H + feat) : 0.f;
    }
    // the ks-1 peer partials of this chunk, all loads in flight together
    float pv[ks - 1][32];
#pragma unroll
    for (int j = 0; j < ks - 1; ++j)
#pragma unroll
      for (int i = 0; i < 32; ++i) pv[j][i] = __ldcg(in0 + (size_t)j * blk + (size_t)i * BM);
    // acc = partial of rank 0, then + rank 1, + rank 2, ... (peer slot of rank s: s, or s-1 past me)
    float acc[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) acc[i] = me == 0 ? __uint_as_float(v[i]) : pv[0][i];
#pragma unroll
    for (int src = 1; src < ks; ++src) {
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float peer = src < me ? pv[src < ks - 1 ? src : ks - 2][i] : pv[src - 1][i];
        acc[i] += src == me ? __uint_as_float(v[i]) : peer;
      }
    }
    if (feat < p.H) {
      // all loads of the chunk precede its first y store: the compiler cannot rule out that y
      // aliases them, and would otherwise wait out each load in turn
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (tc + i < p.T) p.y[(size_t)(tc + i) * p.H + feat] = f32_to_bf16_rn((pmask >> i) & 1u ? acc[i] + dv[i] : acc[i]);
    }
  }
}

__global__ void __launch_bounds__(THREADS, 1)
gemm_lora_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x,
                 const __grid_constant__ CUtensorMap tm_d, const __grid_constant__ CUtensorMap tm_y, GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t s_base = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGE_AREA);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * MAX_STAGES + 2);
  const uint32_t bar_full = smem_u32(bars), bar_empty = bar_full + 8 * MAX_STAGES;
  const uint32_t bar_accum = bar_full + 16 * MAX_STAGES, bar_delta = bar_accum + 8;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.y * BM;
  const int t0 = blockIdx.z * p.BN;
  const int ks = p.ks;                                  // CTAs splitting K (cluster along x)
  const int me = ks > 1 ? (int)cluster_ctarank() : 0;   // this CTA's K slice
  const int kb0 = me * (p.n_kb / ks);                   // first 64-wide K block of the slice
  const int stages = p.stages;
  const int kc = p.kc;                                  // 64-wide K chunks per stage
  const uint32_t xb = (uint32_t)(p.BN * BK * 2);        // one x chunk
  const uint32_t stage_bytes = (uint32_t)kc * (A_BYTES + xb);
  const int nk = p.n_kb / ks / kc;                      // stages' worth of K in this CTA's slice
  const uint32_t ncols = tmem_cols_for(p.BN);

  if (threadIdx.x == 0) {
    for (int s = 0; s < MAX_STAGES; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    mbar_init(bar_accum, 1);
    mbar_init(bar_delta, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_w)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_x)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_d)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_y)) : "memory");
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), ncols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (ks > 1) cluster_sync_all();                       // peers' scratch blocks and barriers exist
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {                                    // TMA producer
      const uint32_t tx = stage_bytes;                  // W tile + x tile
      // When one token tile covers the batch (decode) each W tile is read once; otherwise the
      // CTAs of the other token tiles re-read it, so it must not be marked for early eviction.
      const uint64_t pol_w = (int)gridDim.z == 1 ? policy_evict_first() : policy_evict_last();
      const uint64_t pol_x = policy_evict_last();       // x is re-read by every feature tile
      for (int i = 0; i < nk; ++i) {
        const int s = i % stages;
        const uint32_t ph = (i / stages) & 1;
        if (!mbar_wait(bar_empty + 8 * s, ph ^ 1)) {    // released by every CTA of the cluster
          flag_error(p.err, LORA_DEV_WAIT_TIMEOUT);
          break;
        }
        mbar_arrive_expect_tx(bar_full + 8 * s, tx);
        const uint32_t st = s_base + (uint32_t)s * stage_bytes;
        for (int c = 0; c < kc; ++c) {
          const int kx = (kb0 + i * kc + c) * BK;
          tma_load_2d(st + (uint32_t)c * A_BYTES, &tm_w, kx, m0, bar_full + 8 * s, pol_w);
          tma_load_2d(st + (uint32_t)kc * A_BYTES + (uint32_t)c * xb, &tm_x, kx, t0, bar_full + 8 * s, pol_x);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {                                    // MMA issuer
      const uint32_t idesc = make_idesc_bf16(BM, p.BN);
      for (int i = 0; i < nk; ++i) {
        const int s = i % stages;
        const uint32_t ph = (i / stages) & 1;
        if (!mbar_wait(bar_full + 8 * s, ph)) {
          flag_error(p.err, LORA_DEV_WAIT_TIMEOUT);
          break;
        }
        tc_fence_after();
        const uint32_t st = s_base + (uint32_t)s * stage_bytes;
        for (int c = 0; c < kc; ++c) {
          const uint64_t ad = sw128_kmajor_desc(st + (uint32_t)c * A_BYTES);
          const uint64_t bd = sw128_kmajor_desc(st + (uint32_t)kc * A_BYTES + (uint32_t)c * xb);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)             // 16-element K steps = 32 bytes = 2 descriptor units
            mma_bf16_ss(tmem, ad + 2 * k, bd + 2 * k, idesc, (i | c | k) != 0);
        }
        mma_commit(bar_empty + 8 * s);
      }
      mma_commit(bar_accum);
    }
    __syncwarp();
  }

  // ---- epilogue: all 8 warps ----
  bool ok = mbar_wait(bar_accum, 0);
  if (!ok && lane == 0) flag_error(p.err, LORA_DEV_WAIT_TIMEOUT);
  ok = __syncthreads_and(ok) != 0;
  tc_fence_after();
  const int q = warp & 3, h = warp >> 2;
  const int row = q * 32 + lane;
  const uint32_t tmem_row = tmem + ((uint32_t)(q * 32) << 16);
  if (ks > 1) {
    if (ks == 4)
      split_k_epilogue<4>(p, tmem_row, m0, t0, me, row, lane, h, ok);
    else
      split_k_epilogue<2>(p, tmem_row, m0, t0, me, row, lane, h, ok);
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, ncols);
    cluster_sync_all();                           // no peer may still write into this CTA
    return;
  }
  pdl_wait_then_release();         // the delta and validated ids come from the kernels before this one
  // Stage memory is free now (every load into it belonged to a k-block consumed above):
  // the fp32 delta tile [BN][128] at 0, the bf16 output tile [BN][128] after it (<= 192 KB).
  const uint32_t delta_s = s_base;
  const uint32_t y_s = s_base + (uint32_t)(p.BN * BM * 4);
  const float* delta_p = reinterpret_cast<const float*>(smem);
  uint16_t* y_p = reinterpret_cast<uint16_t*>(smem + (size_t)p.BN * BM * 4);
  if (threadIdx.x == 0 && ok) {
    mbar_arrive_expect_tx(bar_delta, (uint32_t)(p.BN * BM * 4));
    tma_load_2d_plain(delta_s, &tm_d, m0, t0, bar_delta);
  }
  unsigned pm[4];                                 // chunks h + 2k
  presence_masks(p, p.slot, t0, h, 2, p.BN / 32, lane, pm);
  if (ok && !mbar_wait(bar_delta, 0)) {
    flag_error(p.err, LORA_DEV_WAIT_TIMEOUT);
    ok = false;
  }
  ok = __syncthreads_and(ok) != 0;
  if (ok) {
#pragma unroll 1
    for (int k = 0; k < 4; ++k) {
      const int c = h + 2 * k;
      if (c >= p.BN / 32) break;
      uint32_t v[32];
      tmem_ld_32x32b_x32(tmem_row + (uint32_t)(c * 32), v);
      tmem_ld_wait();
      const unsigned pmask = k == 0 ? pm[0] : k == 1 ? pm[1] : k == 2 ? pm[2] : pm[3];
      // y_s[col][feature] bf16 for the TMA store; delta_s[col][feature] fp32 from the TMA load
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const uint32_t col = (uint32_t)(c * 32 + i);
        float acc = __uint_as_float(v[i]);
        if ((pmask >> i) & 1u) acc += delta_p[col * BM + row];
        y_p[col * BM + row] = f32_to_bf16_rn(acc);
      }
    }
    fence_proxy_async_shared();     // generic-proxy writes of y_s -> visible to the TMA store
  }
  __syncthreads();
  if (threadIdx.x == 0 && ok) {
    tma_store_2d(&tm_y, m0, t0, y_s);             // rows past T and features past H are clipped
    bulk_commit_wait_read();                      // the kernel's completion publishes the writes
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, ncols);
}

// ---- persistent variant (batches of more than 256 tokens) ---------------------------------
// One launch serves the n (1 .. LORA_MAX_GROUP) slots of a call that read the same x (q, k and v
// of a layer, or a single slot).  Its tiles are (slot, feature tile, token tile) triples, slot
// major; each CTA walks the tiles c, c + gridDim.x, ...  Within a slot the tiles run in the order
// tile_m / tile_t give, which keeps the smaller of x and W in L2 across waves.  TMEM holds two
// accumulators of BN columns.  Warp 0 issues TMA loads without pause across tile boundaries,
// warp 1 issues the MMAs of tile i into
// accumulator i % 2, and warps 4-7 (one per TMEM lane quarter) drain accumulator (i-1) % 2
// meanwhile: add the delta (read straight from global memory), round to bf16, store y from
// registers.  So a tile's epilogue runs under the next tile's main loop, and one launch for a
// group pays the pipeline fill and the last, unhidden epilogue once instead of once per slot.
// Every tile is computed by the same instruction sequence whichever CTA takes it, so each
// slot's y is bitwise the y of a single-slot launch.
//
// Fused tiles (256-token tiles with at most LORA_TILE_ADAPTERS adapters, planned by the segment
// build): the LoRA term is added inside the accumulator instead of from a delta buffer.  After
// the K blocks of x W^T the tile gets, for each of its adapters b that has LoRA on the slot, the
// K extension
//     acc[n, t] += sum_j B_b[j, n] s_hi[t, j] + sum_j B_b[j, n] s_lo[t, j],    j < r_b rounded up to 16,
// where s = s_hi + s_lo is x A_b for the tile's tokens of adapter b and zero for its other tokens
// (written by the shrink kernel).  Each adapter takes two ring stages: the first holds its B page
// rows for the tile's 128 features (gathered by warps 2-3 with 16-byte cp.async copies into the
// MN-major 128-byte-swizzled layout, a page row's 64-feature half being one 128-byte atom row)
// and the s_hi tile (TMA), the second the s_lo tile (TMA); the MMAs read B_b transposed (MN-major
// A operand).  The epilogue of a fused tile adds no delta: y = bf16(acc), rounded once.  A
// LoRA-only launch (for delta_dbg) runs the extension alone on the fused tiles and writes the
// fp32 accumulator to the debug buffer.
//
// MH = 2: tiles of 256 features.  Each K step issues two M = 128 MMAs that share the stage's x
// tile, into two accumulators of BN columns (all 512 TMEM columns, so one tile at a time: the
// epilogue, now 8 warps, two per lane quarter, is no longer hidden under the next tile), and a
// stage holds 256 W rows.  The shared-memory fill per flop drops by a third (W 32 KB + x 32 KB
// per 64-wide K block for 2 x 128 x 256 x 64 MACs, against 16 + 32 KB for half of them), which
// is what bounds the 128-feature tiles of a prefill-shaped batch.  The LoRA extension gathers
// B rows for both 128-feature blocks of the tile into the stage's W area, one block after the
// other.
struct PersistParams {
  int32_t m_tiles, t_tiles;        // feature tiles; token tiles (per slot)
  int32_t n_ctiles;                // n_group * m_tiles * t_tiles
  int32_t n_group;
  int32_t t_inner;                 // order of a slot's tiles: token tile fastest (see tile_m)
  uint16_t* y[LORA_MAX_GROUP];
  const float* delta[LORA_MAX_GROUP];
  int32_t slot[LORA_MAX_GROUP];
  // fused tiles (tile_plan == nullptr: none)
  const int32_t* tile_plan;
  const uint16_t* pool;
  int64_t num_pages;
  const int32_t* rank;
  int32_t lora_only;               // 1: the LoRA extension alone, fp32 into dbg, fused tiles only
  float* dbg[LORA_MAX_GROUP];
};

// A slot's tile r is (feature tile, token tile).  Consecutive tiles run in one wave of CTAs, so the
// operand whose tiles change fastest is re-read by every wave: with the token tile fastest
// (t_inner, batches of fewer tokens than features) x is re-read and each W tile is taken by all
// token tiles of a wave, so W crosses DRAM once; otherwise W is re-read and x crosses once.  The
// operand re-read is the smaller one, which stays in L2.
__device__ __forceinline__ int tile_m(const PersistParams& pp, int r) { return pp.t_inner ? r / pp.t_tiles : r % pp.m_tiles; }
__device__ __forceinline__ int tile_t(const PersistParams& pp, int r) { return pp.t_inner ? r % pp.t_tiles : r / pp.m_tiles; }

// The LoRA extension of one tile on one slot: -1 when the tile is not fused, else the number of
// the tile's adapters that carry LoRA on the slot, with their page-table rows and ranks.
struct TileLora {
  int nb;
  const int32_t* tab[kTileAdapters];
  int r[kTileAdapters];
  int tmap_b[kTileAdapters];        // the adapter's tile slot: its columns in s_lora
};
__device__ __forceinline__ void tile_lora(const PersistParams& pp, const GemmParams& p, int tile, int slot,
                                          TileLora& L) {
  L.nb = -1;
  if (pp.tile_plan == nullptr) return;
  const int32_t* pl = pp.tile_plan + (size_t)tile * kPlanStride;
  const int n = __ldg(pl);
  if (n < 0) return;
  L.nb = 0;
  for (int b = 0; b < n && b < kTileAdapters; ++b) {
    const int a = __ldg(pl + 1 + b);
    if (a < 0) continue;
    const int r = __ldg(pp.rank + a);
    const int32_t* tab = p.ptab + ((int64_t)a * p.n_slots + slot) * kTabStride;
    if (r < 1 || r > LORA_MAX_RANK || __ldg(tab) < 0) continue;
    L.tab[L.nb] = tab;
    L.r[L.nb] = r;
    L.tmap_b[L.nb] = b;
    ++L.nb;
  }
}
__device__ __forceinline__ int slot_of(const PersistParams& pp, int g) {
  int slot = pp.slot[0];
#pragma unroll
  for (int k = 1; k < LORA_MAX_GROUP; ++k)
    if (g == k) slot = pp.slot[k];
  return slot;
}
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <int MH>
__global__ void __launch_bounds__(THREADS + (MH - 1) * 128, 1)
gemm_lora_persistent(const __grid_constant__ CUtensorMap tm_w0, const __grid_constant__ CUtensorMap tm_w1,
                     const __grid_constant__ CUtensorMap tm_w2, const __grid_constant__ CUtensorMap tm_w3,
                     const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_s0,
                     const __grid_constant__ CUtensorMap tm_s1, const __grid_constant__ CUtensorMap tm_s2,
                     const __grid_constant__ CUtensorMap tm_s3, GemmParams p, PersistParams pp) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t s_base = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGE_AREA);
  // full[MAX_STAGES], empty[MAX_STAGES], tfull[2], tempty[2], wl[MAX_STAGES], go[MAX_STAGES], then
  // the TMEM address
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 4 * MAX_STAGES + 4);
  const uint32_t bar_full = smem_u32(bars), bar_empty = bar_full + 8 * MAX_STAGES;
  const uint32_t bar_tfull = bar_full + 16 * MAX_STAGES, bar_tempty = bar_tfull + 16;
  const uint32_t bar_wl = bar_tempty + 16;              // B page rows of a LoRA stage landed
  // The producer, which waits on every stage's empty barrier in order, tells the loader warps that
  // the ring slot of a LoRA stage is free.  (The loaders skip the base stages, so a parity wait of
  // theirs on the empty barrier could be several phases behind and pass or block wrongly.)
  const uint32_t bar_go = bar_wl + 8 * MAX_STAGES;

  constexpr int TM = MH * BM;                           // features per tile
  constexpr int N_EPI = 4 * MH;                         // epilogue warps
  constexpr int N_ACC = 3 - MH;                         // accumulator buffers (one per tile in flight)
  constexpr uint32_t WB = (uint32_t)MH * A_BYTES;       // W rows of one K chunk
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int stages = p.stages;
  const int kc = p.kc;
  const uint32_t xb = (uint32_t)(p.BN * BK * 2);
  const uint32_t stage_bytes = (uint32_t)kc * (WB + xb);
  const int nk = pp.lora_only ? 0 : p.n_kb / kc;         // base stages per tile
  const uint32_t acc_cols = tmem_cols_for(p.BN);        // one accumulator (MH = 2: one half of the tile)
  const int n_ctas = (int)gridDim.x;
  const int per_slot = pp.m_tiles * pp.t_tiles;
  const bool fused_mode = pp.tile_plan != nullptr;

  if (threadIdx.x == 0) {
    for (int s = 0; s < MAX_STAGES; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
      mbar_init(bar_wl + 8 * s, 2);                     // one arrival per loader warp
      mbar_init(bar_go + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_tfull + 8 * b, 1);
      mbar_init(bar_tempty + 8 * b, N_EPI);             // one arrival per epilogue warp
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_w0)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_x)) : "memory");
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 2 * acc_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {                                    // TMA producer, all tiles back to back
      const uint64_t pol_w = policy_evict_last();       // W tiles are re-read by other token tiles
      const uint64_t pol_x = policy_evict_last();       // x tiles are re-read by other feature tiles
      uint32_t it = 0;
      bool ok = true, waited = false;
      for (int ct = (int)blockIdx.x; ct < pp.n_ctiles && ok; ct += n_ctas) {
        const int g = ct / per_slot, r = ct % per_slot;
        const int m0 = tile_m(pp, r) * TM;
        const int tt = tile_t(pp, r);
        const int t0 = tt * p.BN;
        const CUtensorMap* tw = g == 0 ? &tm_w0 : g == 1 ? &tm_w1 : g == 2 ? &tm_w2 : &tm_w3;
        const CUtensorMap* ts = g == 0 ? &tm_s0 : g == 1 ? &tm_s1 : g == 2 ? &tm_s2 : &tm_s3;
        for (int i = 0; i < nk; ++i, ++it) {
          const int s = it % stages;
          const uint32_t ph = (it / stages) & 1;
          if (!mbar_wait(bar_empty + 8 * s, ph ^ 1)) {
            flag_error(p.err, LORA_DEV_WAIT_TIMEOUT);
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(bar_full + 8 * s, stage_bytes);
          const uint32_t st = s_base + (uint32_t)s * stage_bytes;
          for (int c = 0; c < kc; ++c) {
            const int kx = (i * kc + c) * BK;
#pragma unroll
            for (int h = 0; h < MH; ++h)
              tma_load_2d(st + (uint32_t)c * WB + (uint32_t)h * A_BYTES, tw, kx, m0 + h * BM, bar_full + 8 * s, pol_w);
            tma_load_2d(st + (uint32_t)kc * WB + (uint32_t)c * xb, &tm_x, kx, t0, bar_full + 8 * s, pol_x);
          }
        }
        if (!ok || !fused_mode) continue;
        if (!waited) {                                  // the plan and s come from earlier kernels
          grid_dependency_wait();
          waited = true;
        }
        TileLora TL;
        tile_lora(pp, p, tt, slot_of(pp, g), TL);
        for (int b = 0; b < TL.nb && ok; ++b) {         // s_hi, then s_lo, of adapter b
          for (int part = 0; part < 2; ++part, ++it) {
            const int s = it % stages;
            if (!mbar_wait(bar_empty + 8 * s, ((it / stages) & 1) ^ 1)) {
              flag_error(p.err, LORA_DEV_WAIT_TIMEOUT);
              ok = false;
              break;
            }
            if (part == 0) mbar_arrive(bar_go + 8 * s);     // the loaders may write this slot's B rows
            mbar_arrive_expect_tx(bar_full + 8 * s, xb);
            tma_load_2d(s_base + (uint32_t)s * stage_bytes + WB, ts,
                        TL.tmap_b[b] * 2 * LORA_MAX_RANK + part * LORA_MAX_RANK, t0, bar_full + 8 * s, pol_x);
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {                                    // MMA issuer
      const uint32_t idesc = make_idesc_bf16(BM, p.BN);
      const uint32_t idesc_mn = idesc | kIdescAMnMajor;
      uint32_t it = 0, wl_par = 0;
      int tile = 0;
      bool ok = true, waited = false;
      for (int ct = (int)blockIdx.x; ct < pp.n_ctiles && ok; ct += n_ctas) {
        const int g = ct / per_slot, r = ct % per_slot;
        const int tt = tile_t(pp, r);
        TileLora TL;
        TL.nb = -1;
        if (pp.lora_only) {
          if (!waited) {
            grid_dependency_wait();
            waited = true;
          }
          tile_lora(pp, p, tt, slot_of(pp, g), TL);
          if (TL.nb < 0) continue;                        // the LoRA-only pass skips unfused tiles
        }
        const int b = tile % N_ACC;
        if (!mbar_wait(bar_tempty + 8 * b, ((tile / N_ACC) & 1) ^ 1)) {   // accumulator b drained
          flag_error(p.err, LORA_DEV_WAIT_TIMEOUT);
          break;
        }
        ++tile;
        tc_fence_after();
        const uint32_t acc = tmem + (uint32_t)b * acc_cols;   // MH = 2: b = 0, halves at acc and acc + acc_cols
        for (int i = 0; i < nk; ++i, ++it) {
          const int s = it % stages;
          const uint32_t ph = (it / stages) & 1;
          if (!mbar_wait(bar_full + 8 * s, ph)) {
            flag_error(p.err, LORA_DEV_WAIT_TIMEOUT);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = s_base + (uint32_t)s * stage_bytes;
          for (int c = 0; c < kc; ++c) {
            const uint64_t bd = sw128_kmajor_desc(st + (uint32_t)kc * WB + (uint32_t)c * xb);
#pragma unroll
            for (int k = 0; k < BK / 16; ++k)
#pragma unroll
              for (int h = 0; h < MH; ++h)
                mma_bf16_ss(acc + (uint32_t)h * acc_cols,
                            sw128_kmajor_desc(st + (uint32_t)c * WB + (uint32_t)h * A_BYTES) + 2 * k, bd + 2 * k,
                            idesc, (i | c | k) != 0);
          }
          mma_commit(bar_empty + 8 * s);
        }
        if (fused_mode && !pp.lora_only && ok) {         // the plan is read once the base K blocks are issued
          if (!waited) {
            grid_dependency_wait();
            waited = true;
          }
          tile_lora(pp, p, tt, slot_of(pp, g), TL);
        }
        bool first = nk == 0;                             // LoRA-only: the first MMA starts the sum
        for (int lb = 0; lb < TL.nb && ok; ++lb, it += 2) {
          const int s0 = it % stages, s1 = (it + 1) % stages;
          const uint32_t ph0 = (it / stages) & 1, ph1 = ((it + 1) / stages) & 1;
          const uint32_t wph = (wl_par >> s0) & 1u;
          wl_par ^= 1u << s0;
          if (!mbar_wait(bar_full + 8 * s0, ph0) || !mbar_wait(bar_wl + 8 * s0, wph) ||
              !mbar_wait(bar_full + 8 * s1, ph1)) {
            flag_error(p.err, LORA_DEV_WAIT_TIMEOUT);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st0 = s_base + (uint32_t)s0 * stage_bytes, st1 = s_base + (uint32_t)s1 * stage_bytes;
          const uint64_t bh = sw128_kmajor_desc(st0 + WB), bl = sw128_kmajor_desc(st1 + WB);
          const int n16 = (TL.r[lb] + 15) / 16;
          for (int k = 0; k < n16; ++k) {                 // 16 rank columns: two 8-row groups of B
#pragma unroll
            for (int h = 0; h < MH; ++h) {                // B rows of feature block h at h x A_BYTES
              const uint64_t ad = sw128_mnmajor_desc(st0 + (uint32_t)h * A_BYTES + (uint32_t)k * 4096u, 1024u, 2048u);
              mma_bf16_ss(acc + (uint32_t)h * acc_cols, ad, bh + 2 * k, idesc_mn, first ? 0u : 1u);
              mma_bf16_ss(acc + (uint32_t)h * acc_cols, ad, bl + 2 * k, idesc_mn, 1u);
            }
            first = false;
          }
          mma_commit(bar_empty + 8 * s0);
          mma_commit(bar_empty + 8 * s1);
        }
        if (ok) mma_commit(bar_tfull + 8 * b);            // accumulator b complete
      }
    }
    __syncwarp();
  } else if (warp < 4) {
    // ---- B page rows of the fused tiles' LoRA stages (64 threads) ----
    if (fused_mode) {
      const int l = threadIdx.x - 64;
      grid_dependency_wait();
      uint32_t it = 0, go_par = 0;
      bool ok = true;
      for (int ct = (int)blockIdx.x; ct < pp.n_ctiles && ok; ct += n_ctas) {
        const int g = ct / per_slot, r = ct % per_slot;
        const int m0 = tile_m(pp, r) * TM;
        const int tt = tile_t(pp, r);
        TileLora TL;
        tile_lora(pp, p, tt, slot_of(pp, g), TL);
        it += nk;
        for (int lb = 0; lb < TL.nb && ok; ++lb, it += 2) {
          // chunk c = l + 64 i of a 128-feature block: row j = c / 16 (rank column), 64-feature
          // half h = (c / 8) % 2, 16-byte piece c % 8; page ids are read before the stage is free
          const int r16 = (TL.r[lb] + 15) & ~15;
          int64_t src[16];                                // the page row's start; -1: zero
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int c = l + 64 * i;
            const int j = c >> 4;
            src[i] = -1;                                  // zero: past the rank or a bad page
            if (c < r16 * 16 && j < TL.r[lb]) {
              const int64_t page = __ldg(TL.tab[lb] + LORA_MAX_RANK + j);
              if (page >= 0 && page < pp.num_pages)
                src[i] = page * p.H;
              else
                flag_error(p.err, LORA_DEV_BAD_PAGE);
            }
          }
          const int s = it % stages;
          const uint32_t gph = (go_par >> s) & 1u;
          go_par ^= 1u << s;
          ok = __all_sync(0xffffffffu, mbar_wait(bar_go + 8 * s, gph));
          if (!ok) break;
          const uint32_t st = s_base + (uint32_t)s * stage_bytes;
#pragma unroll
          for (int blk = 0; blk < MH; ++blk)
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int c = l + 64 * i;
              if (c < r16 * 16) {
                const int j = c >> 4, h = (c >> 3) & 1, piece = c & 7;
                const int f = m0 + blk * BM + h * 64 + piece * 8;
                const bool valid = src[i] >= 0 && f < p.H;          // zero past H
                cp_async_16(st + (uint32_t)blk * A_BYTES + (uint32_t)(j >> 3) * 2048u + (uint32_t)h * 1024u +
                                sw128_offset(j, piece),
                            pp.pool + (valid ? src[i] + f : 0), valid);
              }
            }
          cp_async_commit();
          cp_async_wait<0>();
          fence_proxy_async_shared();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_wl + 8 * s);
        }
      }
      if (!ok && lane == 0) flag_error(p.err, LORA_DEV_WAIT_TIMEOUT);
    }
  } else {
    // ---- epilogue warps: TMEM lane quarter q = warp % 4 of feature block hf ----
    const int q = (warp - 4) & 3, hf = (warp - 4) >> 2;
    const int row = hf * BM + q * 32 + lane;
    pdl_wait_then_release();                            // delta, ids and the plan come from earlier kernels
    int tile = 0;
    for (int ct = (int)blockIdx.x; ct < pp.n_ctiles; ct += n_ctas) {
      const int g = ct / per_slot, r = ct % per_slot;
      const int m0 = tile_m(pp, r) * TM;
      const int t0 = tile_t(pp, r) * p.BN;
      const int feat = m0 + row;
      const int slot = slot_of(pp, g);
      TileLora TL;
      TL.nb = -1;
      if (fused_mode) tile_lora(pp, p, tile_t(pp, r), slot, TL);
      if (pp.lora_only && TL.nb < 0) continue;
      const int b = tile % N_ACC;
      const uint32_t tph = (tile / N_ACC) & 1;
      ++tile;
      uint16_t* y = pp.y[0];
      const float* delta = pp.delta[0];
      float* dbg = pp.dbg[0];
#pragma unroll
      for (int k = 1; k < LORA_MAX_GROUP; ++k)
        if (g == k) {
          y = pp.y[k];
          delta = pp.delta[k];
          dbg = pp.dbg[k];
        }
      bool ok = mbar_wait(bar_tfull + 8 * b, tph);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) {
        if (lane == 0) flag_error(p.err, LORA_DEV_WAIT_TIMEOUT);
        break;
      }
      tc_fence_after();
      const uint32_t acc_row = tmem + (uint32_t)(b + hf) * acc_cols + ((uint32_t)(q * 32) << 16);
      const int n_chunks = p.BN / 32;
      for (int c4 = 0; c4 < n_chunks; c4 += 4) {
        unsigned pm[4] = {0u, 0u, 0u, 0u};              // a fused tile's LoRA term is in the accumulator
        if (TL.nb < 0) presence_masks(p, slot, t0, c4, 1, n_chunks, lane, pm);
#pragma unroll 1
        for (int k = 0; k < 4; ++k) {
          const int c = c4 + k;
          if (c >= n_chunks) break;
          const int tc = t0 + c * 32;
          if (tc >= p.T) break;
          uint32_t v[32];
          tmem_ld_32x32b_x32(acc_row + (uint32_t)(c * 32), v);
          tmem_ld_wait();
          if (feat < p.H && pp.lora_only) {
            const bool any = TL.nb > 0;                 // no LoRA stage: the term is zero
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (tc + i < p.T) dbg[(size_t)(tc + i) * p.H + feat] = any ? __uint_as_float(v[i]) : 0.f;
          } else if (feat < p.H) {
            const unsigned pmask = k == 0 ? pm[0] : k == 1 ? pm[1] : k == 2 ? pm[2] : pm[3];
            // every load of the chunk before its first store (y may alias delta as far as the
            // compiler knows)
            float dv[32];
#pragma unroll
            for (int i = 0; i < 32; ++i)
              dv[i] = ((pmask >> i) & 1u) ? __ldg(delta + (size_t)(tc + i) * p.H + feat) : 0.f;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const float a = __uint_as_float(v[i]);
              if (tc + i < p.T) y[(size_t)(tc + i) * p.H + feat] = f32_to_bf16_rn((pmask >> i) & 1u ? a + dv[i] : a);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_tempty + 8 * b);   // accumulator b may be overwritten
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, 2 * acc_cols);
}

// ---- grouped split-K variant (slots that share x, batches of <= 256 tokens) --------------
// One launch serves the n slots of a lora_linear_forward_group call.  Its tiles are (slot,
// feature tile) pairs of 128 features x all BN tokens, K split over a cluster of KS CTAs as in
// gemm_lora_kernel, and persistent clusters walk the tiles.  Warp 0 streams the CTA's K slice
// of W and x for tile after tile, warp 1 accumulates tile i in TMEM accumulator i % 2, and
// warps 4-11 (two per TMEM lane quarter, each taking every other 16-column chunk) finish tile
// i - 1 meanwhile: they write the partial sums of the other owners' token columns to the
// tile's own scratch region, tell each of those owners through an mbarrier in its shared
// memory (one remote arrive per warp, after a cluster-scope fence), wait until the peers have
// done the same for their own columns (cluster-scope acquire), add the KS partials in
// cluster-rank order, add the delta and write y.  So a tile's exchange and epilogue run under
// the next tile's main loop, and the arithmetic is that of gemm_lora_kernel term for term:
// each slot's y is bitwise the y of a single-slot call.
constexpr int GROUP_THREADS = 384;
struct GroupParams {
  uint16_t* y[LORA_MAX_GROUP];
  const float* delta[LORA_MAX_GROUP];
  int32_t slot[LORA_MAX_GROUP];
  int32_t m_tiles;                 // feature tiles per slot
  int32_t n_tiles;                 // (slot, feature tile) pairs
};

template <int KS>
__global__ void __launch_bounds__(GROUP_THREADS, 1)
gemm_lora_group_splitk(const __grid_constant__ CUtensorMap tm_w0, const __grid_constant__ CUtensorMap tm_w1,
                       const __grid_constant__ CUtensorMap tm_w2, const __grid_constant__ CUtensorMap tm_w3,
                       const __grid_constant__ CUtensorMap tm_x, GemmParams p, GroupParams gp) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t s_base = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGE_AREA);
  // full[MAX_STAGES], empty[MAX_STAGES], tfull[2], tempty[2], ready[2], then the TMEM address
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * MAX_STAGES + 6);
  const uint32_t bar_full = smem_u32(bars), bar_empty = bar_full + 8 * MAX_STAGES;
  const uint32_t bar_tfull = bar_full + 16 * MAX_STAGES, bar_tempty = bar_tfull + 16, bar_ready = bar_tempty + 16;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int me = (int)cluster_ctarank();                // this CTA's K slice and token-column owner rank
  const int n_clusters = (int)gridDim.x / KS;
  const int cluster_id = (int)blockIdx.x / KS;
  const int stages = p.stages;
  const int kc = p.kc;
  const uint32_t xb = (uint32_t)(p.BN * BK * 2);
  const uint32_t stage_bytes = (uint32_t)kc * (A_BYTES + xb);
  const int kb0 = me * (p.n_kb / KS);
  const int nk = p.n_kb / KS / kc;
  const uint32_t acc_cols = tmem_cols_for(p.BN);        // one accumulator
  const int w = p.BN / KS;                              // token columns each CTA finishes
  const size_t blk = (size_t)w * BM;                    // one partial block: w columns x 128 features

  if (threadIdx.x == 0) {
    for (int s = 0; s < MAX_STAGES; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_tfull + 8 * b, 1);
      mbar_init(bar_tempty + 8 * b, 8);                 // one arrival per epilogue warp
      mbar_init(bar_ready + 8 * b, (KS - 1) * 8);       // every epilogue warp of every peer
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_w0)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_x)) : "memory");
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 2 * acc_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync_all();                                   // peers' barriers exist before any remote arrive
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {                                    // TMA producer, all tiles back to back
      const uint64_t pol_w = policy_evict_first();      // each W tile is read once
      const uint64_t pol_x = policy_evict_last();       // x is re-read by every tile
      uint32_t it = 0;
      bool ok = true;
      for (int tt = cluster_id; tt < gp.n_tiles && ok; tt += n_clusters) {
        const int g = tt / gp.m_tiles;
        const int m0 = (tt % gp.m_tiles) * BM;
        const CUtensorMap* tw = g == 0 ? &tm_w0 : g == 1 ? &tm_w1 : g == 2 ? &tm_w2 : &tm_w3;
        for (int i = 0; i < nk; ++i, ++it) {
          const int s = it % stages;
          const uint32_t ph = (it / stages) & 1;
          if (!mbar_wait(bar_empty + 8 * s, ph ^ 1)) {
            flag_error(p.err, LORA_DEV_WAIT_TIMEOUT);
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(bar_full + 8 * s, stage_bytes);
          const uint32_t st = s_base + (uint32_t)s * stage_bytes;
          for (int c = 0; c < kc; ++c) {
            const int kx = (kb0 + i * kc + c) * BK;
            tma_load_2d(st + (uint32_t)c * A_BYTES, tw, kx, m0, bar_full + 8 * s, pol_w);
            tma_load_2d(st + (uint32_t)kc * A_BYTES + (uint32_t)c * xb, &tm_x, kx, 0, bar_full + 8 * s, pol_x);
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {                                    // MMA issuer
      const uint32_t idesc = make_idesc_bf16(BM, p.BN);
      uint32_t it = 0;
      int tile = 0;
      bool ok = true;
      for (int tt = cluster_id; tt < gp.n_tiles && ok; tt += n_clusters, ++tile) {
        const int b = tile & 1;
        if (!mbar_wait(bar_tempty + 8 * b, ((tile >> 1) & 1) ^ 1)) {   // accumulator b drained
          flag_error(p.err, LORA_DEV_WAIT_TIMEOUT);
          break;
        }
        tc_fence_after();
        const uint32_t acc = tmem + (uint32_t)b * acc_cols;
        for (int i = 0; i < nk; ++i, ++it) {
          const int s = it % stages;
          const uint32_t ph = (it / stages) & 1;
          if (!mbar_wait(bar_full + 8 * s, ph)) {
            flag_error(p.err, LORA_DEV_WAIT_TIMEOUT);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = s_base + (uint32_t)s * stage_bytes;
          for (int c = 0; c < kc; ++c) {
            const uint64_t ad = sw128_kmajor_desc(st + (uint32_t)c * A_BYTES);
            const uint64_t bd = sw128_kmajor_desc(st + (uint32_t)kc * A_BYTES + (uint32_t)c * xb);
#pragma unroll
            for (int k = 0; k < BK / 16; ++k)
              mma_bf16_ss(acc, ad + 2 * k, bd + 2 * k, idesc, (i | c | k) != 0);
          }
          mma_commit(bar_empty + 8 * s);
        }
        if (ok) mma_commit(bar_tfull + 8 * b);            // accumulator b complete
      }
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ---- epilogue warps: TMEM lane quarter q, 16-column chunks u with u % 2 == h ----
    const int q = warp & 3, h = (warp - 4) >> 2;
    const int row = q * 32 + lane;
    pdl_wait_then_release();      // the delta and ids come from earlier kernels, as do the scratch's last readers
    int tile = 0;
    for (int tt = cluster_id; tt < gp.n_tiles; tt += n_clusters, ++tile) {
      const int b = tile & 1;
      const uint32_t ph = (tile >> 1) & 1;
      const int g = tt / gp.m_tiles;
      const int feat = (tt % gp.m_tiles) * BM + row;    // this thread's output feature
      int slot = gp.slot[0];
      uint16_t* y = gp.y[0];
      const float* delta = gp.delta[0];
#pragma unroll
      for (int k = 1; k < LORA_MAX_GROUP; ++k)
        if (g == k) {
          slot = gp.slot[k];
          y = gp.y[k];
          delta = gp.delta[k];
        }
      bool ok = __all_sync(0xffffffffu, mbar_wait(bar_tfull + 8 * b, ph));
      if (!ok) {
        if (lane == 0) flag_error(p.err, LORA_DEV_WAIT_TIMEOUT);
        break;
      }
      tc_fence_after();
      const uint32_t acc_row = tmem + (uint32_t)b * acc_cols + ((uint32_t)(q * 32) << 16);
      // The tile's scratch region: block (owner o, sender s) at o * (KS - 1) + (s < o ? s : s - 1).
      float* scratch = p.partials + (size_t)tt * KS * (KS - 1) * blk;
      // 1. this CTA's partial sums of the other owners' columns
      for (int u = h; u < p.BN / 16; u += 2) {
        const int o = (u * 16) / w;
        if (o == me) continue;
        uint32_t v[16];
        tmem_ld_32x32b_x16(acc_row + (uint32_t)(u * 16), v);
        tmem_ld_wait();
        float* dst = scratch + (size_t)(o * (KS - 1) + (me < o ? me : me - 1)) * blk + (size_t)(u * 16 - o * w) * BM + row;
#pragma unroll
        for (int i = 0; i < 16; ++i) dst[(size_t)i * BM] = __uint_as_float(v[i]);
      }
      // 2. each of those owners learns that this warp's share of its columns is written: the
      //    warp barrier orders the lanes' stores before lane 0's cluster-scope fence and arrives
      __syncwarp();
      if (lane == 0) {
        asm volatile("fence.acq_rel.cluster;" ::: "memory");
#pragma unroll
        for (int o = 0; o < KS; ++o)
          if (o != me) mbar_arrive_remote_release(bar_ready + 8 * b, (uint32_t)o);
      }
      __syncwarp();
      // 3. own columns [me * w, (me + 1) * w): wait for the peers' partials, add the KS partials
      //    in cluster-rank order, add the delta, write y
      ok = __all_sync(0xffffffffu, mbar_wait_acq_cluster(bar_ready + 8 * b, ph));
      if (!ok) {
        if (lane == 0) flag_error(p.err, LORA_DEV_WAIT_TIMEOUT);
        break;
      }
#pragma unroll 1
      for (int u = me * (w / 16) + h; u < (me + 1) * (w / 16); u += 2) {
        const int tc = u * 16;
        // tokens of this chunk that carry LoRA on the slot (one ballot over the 32-token chunk)
        int a = -1;
        const int tl = (tc & ~31) + lane;
        if (tl < p.T) a = p.tok_adapter[tl];
        const int present = a >= 0 ? p.ptab[((int64_t)a * p.n_slots + slot) * kTabStride] >= 0 : 0;
        const unsigned pmask = __ballot_sync(0xffffffffu, present) >> (tc & 16);
        uint32_t v[16];
        tmem_ld_32x32b_x16(acc_row + (uint32_t)tc, v);
        tmem_ld_wait();
        float dv[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          dv[i] = (((pmask >> i) & 1u) && tc + i < p.T && feat < p.H) ? __ldg(delta + (size_t)(tc + i) * p.H + feat) : 0.f;
        const float* in0 = scratch + (size_t)(me * (KS - 1)) * blk + (size_t)(tc - me * w) * BM + row;
        float pv[KS - 1][16];
#pragma unroll
        for (int j = 0; j < KS - 1; ++j)
#pragma unroll
          for (int i = 0; i < 16; ++i) pv[j][i] = __ldcg(in0 + (size_t)j * blk + (size_t)i * BM);
        float acc[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) acc[i] = me == 0 ? __uint_as_float(v[i]) : pv[0][i];
#pragma unroll
        for (int src = 1; src < KS; ++src) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float peer = src < me ? pv[src < KS - 1 ? src : KS - 2][i] : pv[src - 1][i];
            acc[i] += src == me ? __uint_as_float(v[i]) : peer;
          }
        }
        if (feat < p.H) {
#pragma unroll
          for (int i = 0; i < 16; ++i)
            if (tc + i < p.T) y[(size_t)(tc + i) * p.H + feat] = f32_to_bf16_rn((pmask >> i) & 1u ? acc[i] + dv[i] : acc[i]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_tempty + 8 * b);   // accumulator b may be overwritten
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, 2 * acc_cols);
  cluster_sync_all();                             // no peer may still arrive on this CTA's barriers
}

}  // namespace

namespace {
// Persistent CTAs that can be resident at once (cached per device).
int persistent_ctas() {
  static int cached[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  if (cached[dev] > 0) return cached[dev];
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gemm_lora_persistent<1>, THREADS, SMEM_BYTES) != cudaSuccess ||
      per_sm <= 0) {
    cudaGetLastError();
    per_sm = 1;
  }
  cached[dev] = per_sm * device_sm_count();
  return cached[dev];
}
}  // namespace

namespace {
// Tile geometry of one slot's base GEMM, as launch_gemm and the group launch choose it.
struct Geometry {
  int m_tiles, n_kb, ks, bn, n_tiles, kc, stages;
};
Geometry gemm_geometry(int T, int H, const GemmLaunch& G) {
  Geometry g;
  const int n_sm = device_sm_count();
  g.m_tiles = (H + BM - 1) / BM;
  g.n_kb = H / BK;
  g.ks = 1;
  const int ks_try = g.n_kb % 4 == 0 ? 4 : 2;
  const int bn_try = ((T + 32 * ks_try - 1) / (32 * ks_try)) * (32 * ks_try);
  if (T <= MAX_BN && g.n_kb % 2 == 0 && G.partials &&
      (int64_t)(ks_try - 1) * bn_try * g.m_tiles * BM <= G.partials_floats) {
    // One token tile holds the whole batch (decode): K is split over a cluster of 4 (or 2) CTAs
    // per feature tile instead of cutting the tokens into narrow tiles, so each CTA streams
    // a quarter of W's K range plus the matching quarter of x, and the partial sums meet in
    // the scratch (L2).
    g.ks = ks_try;
    g.bn = bn_try;
    g.n_tiles = 1;
  } else {
    // Token tiles: as few as possible (<= 256 tokens each), but enough to fill about 3/4 of the
    // SMs when the feature tiles alone do not, down to 32-token tiles.
    g.n_tiles = (T + MAX_BN - 1) / MAX_BN;
    const int want = (3 * n_sm / 4 + g.m_tiles - 1) / g.m_tiles;
    const int max_tiles = (T + 31) / 32;
    if (g.n_tiles < want) g.n_tiles = want < max_tiles ? want : max_tiles;
    g.bn = (T + g.n_tiles - 1) / g.n_tiles;
    g.bn = ((g.bn + 31) / 32) * 32;
    if (g.bn > MAX_BN) g.bn = MAX_BN;
    g.n_tiles = (T + g.bn - 1) / g.bn;
  }
  // Each pipeline stage costs a fixed handshake on top of its data, and a CTA's TMA fill rate is
  // bounded, so stages are made large: up to 4 K chunks of 64, at most 96 KB (>= 2 stages).
  const int kb_cta = g.n_kb / g.ks;
  const int chunk_bytes = A_BYTES + g.bn * BK * 2;
  g.kc = 1;                         // wide tiles are MMA-bound: one chunk per stage
  while (g.bn < 128 && g.kc < 4 && 2 * g.kc * chunk_bytes <= 96 * 1024 && kb_cta % (2 * g.kc) == 0) g.kc *= 2;
  g.stages = STAGE_AREA / (g.kc * chunk_bytes);
  if (g.stages > MAX_STAGES) g.stages = MAX_STAGES;
  return g;
}

GemmParams gemm_params(const GemmLaunch& G, const Geometry& g) {
  GemmParams P;
  P.y = G.y;
  P.delta = G.delta;
  P.partials = G.partials;
  P.tok_adapter = G.tok_adapter;
  P.ptab = G.ptab;
  P.err = G.err;
  P.T = G.T;
  P.H = G.H;
  P.BN = g.bn;
  P.n_kb = g.n_kb;
  P.kc = g.kc;
  P.stages = g.stages;
  P.ks = g.ks;
  P.slot = G.slot;
  P.n_slots = G.n_slots;
  return P;
}

// Feature-tile height of a persistent launch: 256-feature tiles (MH = 2) for 256-token tiles when
// their waves cost less.  A 256-feature tile takes about 1.5 times as long as a 128-feature one
// (twice the flops at two thirds of the shared-memory fill per flop, its epilogue not hidden), so
// MH = 2 is taken when 1.5 x its waves is below the waves of 128-feature tiles; a batch whose
// 256-feature tiles leave the last wave nearly empty keeps 128-feature tiles.
int persistent_mh(const Geometry& g, int n, int H) {
  if (g.bn != MAX_BN || g.kc != 1 || g.ks != 1) return 1;
  const int ctas = persistent_ctas();
  const int64_t w1 = ((int64_t)n * g.m_tiles * g.n_tiles + ctas - 1) / ctas;
  const int64_t w2 = ((int64_t)n * ((H + 2 * BM - 1) / (2 * BM)) * g.n_tiles + ctas - 1) / ctas;
  return 3 * w2 < 2 * w1 ? 2 : 1;
}

// One persistent launch over the tiles of the n slots G[0..n) (same x, T and H); with `fused`, the
// plan's fused tiles take their LoRA term in the GEMM (lora_only: that term alone, into lora_dbg).
int launch_persistent(const GemmLaunch* G, int n, const Geometry& g_in, cudaStream_t st, bool fused = false,
                      bool lora_only = false) {
  const int H = G[0].H, T = G[0].T;
  const int mh = persistent_mh(g_in, n, H);
  Geometry g = g_in;
  if (mh == 2) {
    g.m_tiles = (H + 2 * BM - 1) / (2 * BM);
    g.stages = STAGE_AREA / (2 * A_BYTES + g.bn * BK * 2);
  }
  static DeviceFlags attr1, attr2;
  int rc = mh == 1 ? ensure_smem_attr(attr1, gemm_lora_persistent<1>, SMEM_BYTES, "gemm kernel attribute")
                   : ensure_smem_attr(attr2, gemm_lora_persistent<2>, SMEM_BYTES, "gemm kernel attribute");
  if (rc != LORA_OK) return rc;
  CUtensorMap tm_w[LORA_MAX_GROUP], tm_x;
  for (int i = 0; i < n; ++i) {
    rc = encode_2d(&tm_w[i], G[i].W, (uint64_t)H, (uint64_t)H, (uint32_t)BM);
    if (rc != LORA_OK) return rc;
  }
  for (int i = n; i < LORA_MAX_GROUP; ++i) tm_w[i] = tm_w[0];
  rc = encode_2d(&tm_x, G[0].x, (uint64_t)H, (uint64_t)T, (uint32_t)g.bn);
  if (rc != LORA_OK) return rc;
  CUtensorMap tm_s[LORA_MAX_GROUP];
  for (int i = 0; i < LORA_MAX_GROUP; ++i) {
    if (fused && i < n) {
      rc = encode_2d(&tm_s[i], G[i].s_lora, (uint64_t)kSCols, (uint64_t)T, (uint32_t)g.bn);
      if (rc != LORA_OK) return rc;
    } else {
      tm_s[i] = tm_x;                                   // never read
    }
  }
  PersistParams pp = {};
  pp.m_tiles = g.m_tiles;
  pp.t_tiles = g.n_tiles;
  pp.n_group = n;
  pp.t_inner = T < H ? 1 : 0;                           // x smaller than W: keep x in L2
  pp.n_ctiles = n * g.m_tiles * g.n_tiles;
  for (int i = 0; i < LORA_MAX_GROUP; ++i) {
    const int j = i < n ? i : 0;
    pp.y[i] = G[j].y;
    pp.delta[i] = G[j].delta;
    pp.slot[i] = G[j].slot;
    pp.dbg[i] = G[j].lora_dbg;
  }
  if (fused) {
    pp.tile_plan = G[0].tile_plan;
    pp.pool = G[0].pool;
    pp.num_pages = G[0].num_pages;
    pp.rank = G[0].rank;
    pp.lora_only = lora_only ? 1 : 0;
  }
  int ctas = persistent_ctas();
  if (ctas > pp.n_ctiles) ctas = pp.n_ctiles;
  cudaError_t e;
  {
    ProfScope prof(G[0].prof, LORA_KIND_GEMM, st);
    e = mh == 1 ? launch_pdl(G[0].pdl, gemm_lora_persistent<1>, dim3(ctas), dim3(THREADS), SMEM_BYTES, st, tm_w[0],
                             tm_w[1], tm_w[2], tm_w[3], tm_x, tm_s[0], tm_s[1], tm_s[2], tm_s[3], gemm_params(G[0], g), pp)
                : launch_pdl(G[0].pdl, gemm_lora_persistent<2>, dim3(ctas), dim3(THREADS + 128), SMEM_BYTES, st,
                             tm_w[0], tm_w[1], tm_w[2], tm_w[3], tm_x, tm_s[0], tm_s[1], tm_s[2], tm_s[3],
                             gemm_params(G[0], g), pp);
    if (e == cudaSuccess) e = cudaGetLastError();
  }
  return e == cudaSuccess ? LORA_OK : lora_cuda_fail(e, "gemm_lora_persistent launch");
}
}  // namespace

int launch_gemm(const GemmLaunch& G, cudaStream_t st) {
  const Geometry g = gemm_geometry(G.T, G.H, G);
  // More tiles than resident CTAs: persistent CTAs overlap each tile's epilogue with the next
  // tile's main loop.
  if (g.ks == 1 && g.m_tiles * g.n_tiles > persistent_ctas()) return launch_persistent(&G, 1, g, st);
  static DeviceFlags attr;
  int rc = ensure_smem_attr(attr, gemm_lora_kernel, SMEM_BYTES, "gemm kernel attribute");
  if (rc != LORA_OK) return rc;
  const int ep_rows = g.bn / g.ks;  // token rows of the delta and y tiles one CTA's epilogue moves
  CUtensorMap tm_w, tm_x, tm_d, tm_y;
  rc = encode_2d(&tm_w, G.W, (uint64_t)G.H, (uint64_t)G.H, (uint32_t)BM);
  if (rc != LORA_OK) return rc;
  rc = encode_2d(&tm_x, G.x, (uint64_t)G.H, (uint64_t)G.T, (uint32_t)g.bn);
  if (rc != LORA_OK) return rc;
  // The delta tile the epilogue adds and the output tile it writes: [bn tokens][128 features].
  rc = encode_2d_plain(&tm_d, G.delta, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, (uint64_t)G.H, (uint64_t)G.T, (uint32_t)ep_rows);
  if (rc != LORA_OK) return rc;
  rc = encode_2d_plain(&tm_y, G.y, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)G.H, (uint64_t)G.T, (uint32_t)ep_rows);
  if (rc != LORA_OK) return rc;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(g.ks, g.m_tiles, g.n_tiles);
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = st;
  cudaLaunchAttribute attrs[2];
  attrs[0].id = cudaLaunchAttributeClusterDimension;
  attrs[0].val.clusterDim.x = g.ks;
  attrs[0].val.clusterDim.y = 1;
  attrs[0].val.clusterDim.z = 1;
  attrs[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = G.pdl ? 2 : 1;
  cudaError_t e;
  {
    ProfScope prof(G.prof, LORA_KIND_GEMM, st);
    e = cudaLaunchKernelEx(&cfg, gemm_lora_kernel, tm_w, tm_x, tm_d, tm_y, gemm_params(G, g));
    if (e == cudaSuccess) e = cudaGetLastError();
  }
  return e == cudaSuccess ? LORA_OK : lora_cuda_fail(e, "gemm_lora_kernel launch");
}

namespace {
// Split-K geometry of a batch of <= 256 tokens, as launch_gemm chooses it.
struct SplitK {
  int ks, bn, kc, stages;
};
bool split_k_geometry(int T, int H, SplitK& g) {
  const int n_kb = H / BK;
  if (T > MAX_BN || n_kb % 2 != 0) return false;
  g.ks = n_kb % 4 == 0 ? 4 : 2;
  g.bn = ((T + 32 * g.ks - 1) / (32 * g.ks)) * (32 * g.ks);
  const int kb_cta = n_kb / g.ks;
  const int chunk_bytes = A_BYTES + g.bn * BK * 2;
  g.kc = 1;
  while (g.bn < 128 && g.kc < 4 && 2 * g.kc * chunk_bytes <= 96 * 1024 && kb_cta % (2 * g.kc) == 0) g.kc *= 2;
  g.stages = STAGE_AREA / (g.kc * chunk_bytes);
  if (g.stages > MAX_STAGES) g.stages = MAX_STAGES;
  return true;
}

template <int KS>
int group_clusters() {
  static int cached[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  if (cached[dev] > 0) return cached[dev];
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(KS * 64);
  cfg.blockDim = dim3(GROUP_THREADS);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = KS;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, gemm_lora_group_splitk<KS>, &cfg) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    n = device_sm_count() / KS;
  }
  cached[dev] = n;
  return n;
}

template <int KS>
int launch_group_ks(const GemmLaunch* G, int n, const SplitK& sk, cudaStream_t st) {
  static DeviceFlags attr;
  int rc0 = ensure_smem_attr(attr, gemm_lora_group_splitk<KS>, SMEM_BYTES, "gemm group kernel attribute");
  if (rc0 != LORA_OK) return rc0;
  const int H = G[0].H, T = G[0].T;
  const int m_tiles = (H + BM - 1) / BM;
  CUtensorMap tm_w[LORA_MAX_GROUP], tm_x;
  for (int i = 0; i < n; ++i) {
    int rc = encode_2d(&tm_w[i], G[i].W, (uint64_t)H, (uint64_t)H, (uint32_t)BM);
    if (rc != LORA_OK) return rc;
  }
  for (int i = n; i < LORA_MAX_GROUP; ++i) tm_w[i] = tm_w[0];
  int rc = encode_2d(&tm_x, G[0].x, (uint64_t)H, (uint64_t)T, (uint32_t)sk.bn);
  if (rc != LORA_OK) return rc;
  GemmParams P;
  P.y = G[0].y;
  P.delta = G[0].delta;
  P.partials = G[0].partials;
  P.tok_adapter = G[0].tok_adapter;
  P.ptab = G[0].ptab;
  P.err = G[0].err;
  P.T = T;
  P.H = H;
  P.BN = sk.bn;
  P.n_kb = H / BK;
  P.kc = sk.kc;
  P.stages = sk.stages;
  P.ks = KS;
  P.slot = G[0].slot;
  P.n_slots = G[0].n_slots;
  GroupParams gp = {};
  for (int i = 0; i < LORA_MAX_GROUP; ++i) {
    const int j = i < n ? i : 0;
    gp.y[i] = G[j].y;
    gp.delta[i] = G[j].delta;
    gp.slot[i] = G[j].slot;
  }
  gp.m_tiles = m_tiles;
  gp.n_tiles = n * m_tiles;
  int clusters = group_clusters<KS>();
  if (clusters > gp.n_tiles) clusters = gp.n_tiles;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(clusters * KS);
  cfg.blockDim = dim3(GROUP_THREADS);
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
  cfg.numAttrs = G[0].pdl ? 2 : 1;
  cudaError_t e;
  {
    ProfScope prof(G[0].prof, LORA_KIND_GEMM, st);
    e = cudaLaunchKernelEx(&cfg, gemm_lora_group_splitk<KS>, tm_w[0], tm_w[1], tm_w[2], tm_w[3], tm_x, P, gp);
    if (e == cudaSuccess) e = cudaGetLastError();
  }
  return e == cudaSuccess ? LORA_OK : lora_cuda_fail(e, "gemm_lora_group_splitk launch");
}
}  // namespace

namespace {
bool same_input(const GemmLaunch* G, int n) {
  for (int i = 1; i < n; ++i)
    if (G[i].x != G[0].x || G[i].T != G[0].T || G[i].H != G[0].H || G[i].partials != G[0].partials) return false;
  return true;
}
// The group's split-K launch (batches of <= 256 tokens): geometry and scratch for n slots.
bool group_split_fits(const GemmLaunch* G, int n, SplitK& sk) {
  if (!split_k_geometry(G[0].T, G[0].H, sk)) return false;
  const int m_tiles = (G[0].H + BM - 1) / BM;
  return G[0].partials && (int64_t)n * (sk.ks - 1) * sk.bn * m_tiles * BM <= G[0].partials_floats;
}
}  // namespace

bool gemm_group_fits(const GemmLaunch* G, int n) {
  if (n < 2 || n > LORA_MAX_GROUP || !same_input(G, n)) return false;
  SplitK sk;
  if (group_split_fits(G, n, sk)) return true;
  return gemm_geometry(G[0].T, G[0].H, G[0]).ks == 1;     // larger batches: one persistent launch
}

bool gemm_fused_fits(const GemmLaunch* G, int n) {
  if (n < 1 || n > LORA_MAX_GROUP || !same_input(G, n) || !G[0].tile_plan || G[0].T <= kTileTokens) return false;
  const Geometry g = gemm_geometry(G[0].T, G[0].H, G[0]);
  if (g.ks != 1 || g.bn != kTileTokens || g.kc != 1 || g.n_kb < kShrinkCluster) return false;
  // a single slot keeps the one-wave kernel when its tiles fit the GPU at once
  return n > 1 || g.m_tiles * g.n_tiles > persistent_ctas();
}

int launch_gemm_fused(const GemmLaunch* G, int n, bool lora_only, cudaStream_t st) {
  if (!gemm_fused_fits(G, n)) return lora_fail(LORA_EINVAL, "launch_gemm_fused: batch geometry without fused tiles");
  return launch_persistent(G, n, gemm_geometry(G[0].T, G[0].H, G[0]), st, true, lora_only);
}

int launch_gemm_group(const GemmLaunch* G, int n, cudaStream_t st) {
  if (!gemm_group_fits(G, n)) return lora_fail(LORA_EINVAL, "launch_gemm_group: the slots do not form a group");
  SplitK sk;
  if (group_split_fits(G, n, sk))
    return sk.ks == 4 ? launch_group_ks<4>(G, n, sk, st) : launch_group_ks<2>(G, n, sk, st);
  return launch_persistent(G, n, gemm_geometry(G[0].T, G[0].H, G[0]), st);
}
