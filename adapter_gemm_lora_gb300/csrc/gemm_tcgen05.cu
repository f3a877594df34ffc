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
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "lora_internal.h"

namespace {

constexpr int BM = 128;          // output features per tile (MMA M)
constexpr int BK = 64;           // K elements per stage: one 128-byte swizzle atom wide
constexpr int MAX_BN = 256;      // tokens per tile (MMA N)
constexpr int MAX_STAGES = 8;
constexpr int A_BYTES = BM * BK * 2;
constexpr int STAGE_AREA = 192 * 1024;        // ring of stages; reused by the epilogue
constexpr int BAR_BYTES = 256;
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

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void flag_error(int32_t* err, int32_t bits) {
  atomicCAS(err, 0, LORA_EDEVICE);
  atomicOr(err + 1, bits);
}

// ---- mbarrier ---------------------------------------------------------------------------
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
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(1000000u)   // suspend-time hint (ns); the phase completing wakes it
      : "memory");
  return ok != 0;
}
// Wait for the phase of the given parity to complete; false if the wait runs out.  The bound
// is counted with the SM's own cycle counter (clock64): it is cheap to read, unlike the global
// timer, whose read latency would otherwise land on every pipeline step.  4e9 cycles is about
// 2 s at the maximum SM clock.
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

// ---- TMA --------------------------------------------------------------------------------
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1, uint32_t bar,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar), "l"(policy)
      : "memory");
}
__device__ __forceinline__ void tma_load_2d_plain(uint32_t dst, const CUtensorMap* map, int c0, int c1, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, int c0, int c1, uint32_t src) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1), "r"(src)
               : "memory");
}
__device__ __forceinline__ void fence_proxy_async_shared() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ---- clusters and programmatic dependent launch --------------------------------------------
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// ---- tcgen05 ----------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void mma_bf16_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive once on `bar` when every MMA this thread issued so far has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// 32 lanes x 32 consecutive columns of 32-bit TMEM data: thread i gets lane (base + i).
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
// 32 lanes x 16 consecutive columns.
__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor for a K-major operand tile written by TMA with the
// 128-byte swizzle: rows of 64 bf16 (128 B), 8-row groups 1024 B apart.
__device__ __forceinline__ uint64_t sw128_kmajor_desc(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4)   // start address, 16-byte units
         | ((uint64_t)1 << 16)                  // leading-dimension byte offset (unused here)
         | ((uint64_t)(1024 >> 4) << 32)        // stride-dimension byte offset: 8 rows x 128 B
         | ((uint64_t)1 << 46)                  // descriptor version for tcgen05
         | ((uint64_t)2 << 61);                 // swizzle mode: 128-byte
}

// Instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B, both K-major.
__host__ __device__ constexpr uint32_t make_idesc_bf16(int M, int N) {
  return (1u << 4)                           // D format: f32
         | (1u << 7)                         // A format: bf16
         | (1u << 10)                        // B format: bf16
         | ((uint32_t)(N >> 3) << 17)        // N / 8
         | ((uint32_t)(M >> 4) << 24);       // M / 16
}

__host__ __device__ inline uint32_t tmem_cols_for(int bn) {
  uint32_t c = 32;
  while ((int)c < bn) c <<= 1;
  return c;
}

__device__ __forceinline__ uint16_t f32_to_bf16_rn(float v) { return __bfloat16_as_ushort(__float2bfloat16_rn(v)); }

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

__device__ __forceinline__ void bulk_commit_wait_read() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
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
// of a layer, or a single slot).  Its tiles are (slot, token tile, feature tile) triples, slot
// major; each CTA walks the tiles c, c + gridDim.x, ...  Consecutive tiles are consecutive
// feature tiles of one token tile, so the CTAs of a wave share x tiles in L2, and a slot's W
// stays in L2 while its tiles are in flight.  TMEM holds two accumulators of BN columns.  Warp 0
// issues TMA loads without pause across tile boundaries, warp 1 issues the MMAs of tile i into
// accumulator i % 2, and warps 4-7 (one per TMEM lane quarter) drain accumulator (i-1) % 2
// meanwhile: add the delta (read straight from global memory), round to bf16, store y from
// registers.  So a tile's epilogue runs under the next tile's main loop, and one launch for a
// group pays the pipeline fill and the last, unhidden epilogue once instead of once per slot.
// Every tile is computed by the same instruction sequence whichever CTA takes it, so each
// slot's y is bitwise the y of a single-slot launch.
struct PersistParams {
  int32_t m_tiles, t_tiles;        // feature tiles; token tiles (per slot)
  int32_t n_ctiles;                // n_group * m_tiles * t_tiles
  int32_t n_group;
  uint16_t* y[LORA_MAX_GROUP];
  const float* delta[LORA_MAX_GROUP];
  int32_t slot[LORA_MAX_GROUP];
};

__global__ void __launch_bounds__(THREADS, 1)
gemm_lora_persistent(const __grid_constant__ CUtensorMap tm_w0, const __grid_constant__ CUtensorMap tm_w1,
                     const __grid_constant__ CUtensorMap tm_w2, const __grid_constant__ CUtensorMap tm_w3,
                     const __grid_constant__ CUtensorMap tm_x, GemmParams p, PersistParams pp) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t s_base = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGE_AREA);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * MAX_STAGES + 4);
  const uint32_t bar_full = smem_u32(bars), bar_empty = bar_full + 8 * MAX_STAGES;
  const uint32_t bar_tfull = bar_full + 16 * MAX_STAGES, bar_tempty = bar_tfull + 16;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int stages = p.stages;
  const int kc = p.kc;
  const uint32_t xb = (uint32_t)(p.BN * BK * 2);
  const uint32_t stage_bytes = (uint32_t)kc * (A_BYTES + xb);
  const int nk = p.n_kb / kc;
  const uint32_t acc_cols = tmem_cols_for(p.BN);        // one accumulator
  const int n_ctas = (int)gridDim.x;
  const int per_slot = pp.m_tiles * pp.t_tiles;

  if (threadIdx.x == 0) {
    for (int s = 0; s < MAX_STAGES; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_tfull + 8 * b, 1);
      mbar_init(bar_tempty + 8 * b, 4);                 // one arrival per epilogue warp
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
      bool ok = true;
      for (int ct = (int)blockIdx.x; ct < pp.n_ctiles && ok; ct += n_ctas) {
        const int g = ct / per_slot, r = ct % per_slot;
        const int m0 = (r % pp.m_tiles) * BM;
        const int t0 = (r / pp.m_tiles) * p.BN;
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
            const int kx = (i * kc + c) * BK;
            tma_load_2d(st + (uint32_t)c * A_BYTES, tw, kx, m0, bar_full + 8 * s, pol_w);
            tma_load_2d(st + (uint32_t)kc * A_BYTES + (uint32_t)c * xb, &tm_x, kx, t0, bar_full + 8 * s, pol_x);
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
      for (int ct = (int)blockIdx.x; ct < pp.n_ctiles && ok; ct += n_ctas, ++tile) {
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
    // ---- epilogue warps: TMEM lane quarter q = warp - 4 ----
    const int q = warp - 4;
    const int row = q * 32 + lane;
    pdl_wait_then_release();                            // delta and ids come from earlier kernels
    int tile = 0;
    for (int ct = (int)blockIdx.x; ct < pp.n_ctiles; ct += n_ctas, ++tile) {
      const int b = tile & 1;
      const int g = ct / per_slot, r = ct % per_slot;
      const int m0 = (r % pp.m_tiles) * BM;
      const int t0 = (r / pp.m_tiles) * p.BN;
      const int feat = m0 + row;
      int slot = pp.slot[0];
      uint16_t* y = pp.y[0];
      const float* delta = pp.delta[0];
#pragma unroll
      for (int k = 1; k < LORA_MAX_GROUP; ++k)
        if (g == k) {
          slot = pp.slot[k];
          y = pp.y[k];
          delta = pp.delta[k];
        }
      bool ok = mbar_wait(bar_tfull + 8 * b, (tile >> 1) & 1);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) {
        if (lane == 0) flag_error(p.err, LORA_DEV_WAIT_TIMEOUT);
        break;
      }
      tc_fence_after();
      const uint32_t acc_row = tmem + (uint32_t)b * acc_cols + ((uint32_t)(q * 32) << 16);
      const int n_chunks = p.BN / 32;
      for (int c4 = 0; c4 < n_chunks; c4 += 4) {
        unsigned pm[4];
        presence_masks(p, slot, t0, c4, 1, n_chunks, lane, pm);
#pragma unroll 1
        for (int k = 0; k < 4; ++k) {
          const int c = c4 + k;
          if (c >= n_chunks) break;
          const int tc = t0 + c * 32;
          if (tc >= p.T) break;
          uint32_t v[32];
          tmem_ld_32x32b_x32(acc_row + (uint32_t)(c * 32), v);
          tmem_ld_wait();
          const unsigned pmask = k == 0 ? pm[0] : k == 1 ? pm[1] : k == 2 ? pm[2] : pm[3];
          if (feat < p.H) {
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

// Arrive on the mbarrier at `local_bar`'s offset in CTA `rank` of the cluster, with cluster-scope
// release: this thread's earlier writes, global memory included, are visible to any thread of
// the cluster whose acquire wait observes the phase the arrival completes.
__device__ __forceinline__ void mbar_arrive_remote_release(uint32_t local_bar, uint32_t rank) {
  uint32_t rb;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(rb) : "r"(local_bar), "r"(rank));
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(rb) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_acq_cluster(uint32_t bar, uint32_t parity) {
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
// Bounded like mbar_wait.
__device__ __forceinline__ bool mbar_wait_acq_cluster(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait_acq_cluster(bar, parity)) return true;
  const long long c0 = clock64();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait_acq_cluster(bar, parity)) return true;
    if (clock64() - c0 > kWaitLimitCycles) return false;
  }
}

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

// ---- host side --------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// 2-D bf16 tensor [rows][inner] row-major, box = box_rows x 64 elements, 128-byte swizzle.
int encode_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint32_t box_rows) {
  auto fn = get_encode_fn();
  if (!fn) return lora_fail(LORA_ECUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {inner * 2};
  const cuuint32_t box[2] = {(cuuint32_t)BK, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return lora_fail(LORA_ECUDA, "cuTensorMapEncodeTiled failed with code " + std::to_string((int)r));
  return LORA_OK;
}

// 2-D tensor [rows][inner] row-major without swizzle, box = box_rows x 128 elements.
int encode_2d_plain(CUtensorMap* map, const void* base, CUtensorMapDataType dt, uint32_t esize, uint64_t inner,
                    uint64_t rows, uint32_t box_rows) {
  auto fn = get_encode_fn();
  if (!fn) return lora_fail(LORA_ECUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {inner * esize};
  const cuuint32_t box[2] = {(cuuint32_t)BM, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return lora_fail(LORA_ECUDA, "cuTensorMapEncodeTiled failed with code " + std::to_string((int)r));
  return LORA_OK;
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
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gemm_lora_persistent, THREADS, SMEM_BYTES) != cudaSuccess ||
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

// One persistent launch over the tiles of the n slots G[0..n) (same x, T and H).
int launch_persistent(const GemmLaunch* G, int n, const Geometry& g, cudaStream_t st) {
  static DeviceFlags attr;
  int rc = ensure_smem_attr(attr, gemm_lora_persistent, SMEM_BYTES, "gemm kernel attribute");
  if (rc != LORA_OK) return rc;
  const int H = G[0].H, T = G[0].T;
  CUtensorMap tm_w[LORA_MAX_GROUP], tm_x;
  for (int i = 0; i < n; ++i) {
    rc = encode_2d(&tm_w[i], G[i].W, (uint64_t)H, (uint64_t)H, (uint32_t)BM);
    if (rc != LORA_OK) return rc;
  }
  for (int i = n; i < LORA_MAX_GROUP; ++i) tm_w[i] = tm_w[0];
  rc = encode_2d(&tm_x, G[0].x, (uint64_t)H, (uint64_t)T, (uint32_t)g.bn);
  if (rc != LORA_OK) return rc;
  PersistParams pp = {};
  pp.m_tiles = g.m_tiles;
  pp.t_tiles = g.n_tiles;
  pp.n_group = n;
  pp.n_ctiles = n * g.m_tiles * g.n_tiles;
  for (int i = 0; i < LORA_MAX_GROUP; ++i) {
    const int j = i < n ? i : 0;
    pp.y[i] = G[j].y;
    pp.delta[i] = G[j].delta;
    pp.slot[i] = G[j].slot;
  }
  int ctas = persistent_ctas();
  if (ctas > pp.n_ctiles) ctas = pp.n_ctiles;
  cudaError_t e = launch_pdl(G[0].pdl, gemm_lora_persistent, dim3(ctas), dim3(THREADS), SMEM_BYTES, st, tm_w[0],
                             tm_w[1], tm_w[2], tm_w[3], tm_x, gemm_params(G[0], g), pp);
  if (e == cudaSuccess) e = cudaGetLastError();
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
  cudaError_t e = cudaLaunchKernelEx(&cfg, gemm_lora_kernel, tm_w, tm_x, tm_d, tm_y, gemm_params(G, g));
  if (e == cudaSuccess) e = cudaGetLastError();
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
  cudaError_t e = cudaLaunchKernelEx(&cfg, gemm_lora_group_splitk<KS>, tm_w[0], tm_w[1], tm_w[2], tm_w[3], tm_x, P, gp);
  if (e == cudaSuccess) e = cudaGetLastError();
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

int launch_gemm_group(const GemmLaunch* G, int n, cudaStream_t st) {
  if (!gemm_group_fits(G, n)) return lora_fail(LORA_EINVAL, "launch_gemm_group: the slots do not form a group");
  SplitK sk;
  if (group_split_fits(G, n, sk))
    return sk.ks == 4 ? launch_group_ks<4>(G, n, sk, st) : launch_group_ks<2>(G, n, sk, st);
  return launch_persistent(G, n, gemm_geometry(G[0].T, G[0].H, G[0]), st);
}
