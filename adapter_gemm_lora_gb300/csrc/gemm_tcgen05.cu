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
// Per CTA: one 128 x BN output tile over a slice of K.  Warp 0 issues TMA loads into a
// 4-stage ring, warp 1 owns TMEM and a single thread issues the MMAs, then all 8 warps
// drain TMEM (warp w reads TMEM lanes 32*(w%4) .. +31, half the columns each).
// Small grids (decode batches: H/128 x 1 tiles for 152 SMs) split K over the CTAs of a
// thread-block cluster; each CTA then owns BN/ks token columns, receives the other CTAs'
// fp32 partials for them through distributed shared memory, and sums them in split order
// (deterministic) before the epilogue.  The mainloop reads only x and W, so the kernel is
// launched as a programmatic dependent of the LoRA kernels before it and waits for them
// (griddepcontrol.wait) only before its epilogue reads the delta.
// Every mbarrier wait is bounded (~2 s); on expiry the CTA raises the device error word,
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
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = MAX_BN * BK * 2;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int BAR_BYTES = 256;
constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + BAR_BYTES;
constexpr int THREADS = 256;
constexpr uint64_t kWaitLimitNs = 2000000000ull;

struct GemmParams {
  uint16_t* y;
  const float* delta;
  const int32_t* tok_adapter;
  const int32_t* ptab;
  int32_t* err;
  int32_t T, H, BN, n_kb, ks, slot, n_slots;
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
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Wait for the phase of the given parity to complete; false if ~2 s pass first.
__device__ __noinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (true) {
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 > kWaitLimitNs) return false;
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
__device__ __forceinline__ void bulk_commit_and_wait_all() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_shared() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void st_shared_u16(uint32_t addr, uint16_t v) {
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}
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
// Address of the same shared-memory offset in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t map_to_cta(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ float ld_shared_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
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

__global__ void __launch_bounds__(THREADS, 1)
gemm_lora_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x,
                 const __grid_constant__ CUtensorMap tm_d, const __grid_constant__ CUtensorMap tm_y, GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t s_base = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 2);
  const uint32_t bar_full = smem_u32(bars), bar_empty = bar_full + 8 * STAGES, bar_accum = bar_full + 16 * STAGES;
  const uint32_t bar_delta = bar_accum + 8;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = blockIdx.x;                     // == rank in the (ks, 1, 1) cluster
  const int m0 = blockIdx.y * BM;
  const int t0 = blockIdx.z * p.BN;
  const int kb0 = split * p.n_kb / p.ks, kb1 = (split + 1) * p.n_kb / p.ks;
  const int nk = kb1 - kb0;
  const uint32_t ncols = tmem_cols_for(p.BN);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
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
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {                                  // TMA producer
      const uint32_t tx = A_BYTES + (uint32_t)p.BN * BK * 2;
      // With one token tile (decode batches) W streams through once; otherwise every token tile
      // re-reads it, so it must not be marked for early eviction.
      const uint64_t pol_w = gridDim.z == 1 ? policy_evict_first() : policy_evict_last();
      const uint64_t pol_x = policy_evict_last();     // x is re-read by every feature tile
      for (int i = 0; i < nk; ++i) {
        const int s = i % STAGES;
        const uint32_t ph = (i / STAGES) & 1;
        if (!mbar_wait(bar_empty + 8 * s, ph ^ 1)) {
          flag_error(p.err, LORA_DEV_WAIT_TIMEOUT);
          break;
        }
        mbar_arrive_expect_tx(bar_full + 8 * s, tx);
        const int kc = (kb0 + i) * BK;
        tma_load_2d(s_base + s * STAGE_BYTES, &tm_w, kc, m0, bar_full + 8 * s, pol_w);
        tma_load_2d(s_base + s * STAGE_BYTES + A_BYTES, &tm_x, kc, t0, bar_full + 8 * s, pol_x);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {                                  // MMA issuer
      const uint32_t idesc = make_idesc_bf16(BM, p.BN);
      for (int i = 0; i < nk; ++i) {
        const int s = i % STAGES;
        const uint32_t ph = (i / STAGES) & 1;
        if (!mbar_wait(bar_full + 8 * s, ph)) {
          flag_error(p.err, LORA_DEV_WAIT_TIMEOUT);
          break;
        }
        tc_fence_after();
        const uint64_t ad = sw128_kmajor_desc(s_base + s * STAGE_BYTES);
        const uint64_t bd = sw128_kmajor_desc(s_base + s * STAGE_BYTES + A_BYTES);
#pragma unroll
        for (int k = 0; k < BK / 16; ++k)             // 16-element K steps = 32 bytes = 2 descriptor units
          mma_bf16_ss(tmem, ad + 2 * k, bd + 2 * k, idesc, (i | k) != 0);
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
  pdl_wait_then_release();         // the delta and validated ids come from the kernels before this one
  const int q = warp & 3, h = warp >> 2;
  const int row = q * 32 + lane;
  const int n = m0 + row;
  const int cols = p.BN / p.ks;     // token columns this CTA finishes
  // Stage memory is free now.  Layout: [0, BN*512) fp32 partials received from the cluster,
  // [ks][cols][128]; this CTA's own slot in it (never written by peers) holds the fp32 delta
  // sub-tile [cols][128]; the bf16 output sub-tile [cols][128] follows at BN*512 (<= 160 KB).
  const uint32_t recv = s_base;
  const uint32_t delta_s = s_base + (uint32_t)(split * cols * BM * 4);
  const uint32_t y_s = s_base + (uint32_t)(p.BN * BM * 4);
  const uint32_t tmem_row = tmem + ((uint32_t)(q * 32) << 16);
  const int tc0 = t0 + split * cols;                 // first token column this CTA finishes
  if (threadIdx.x == 0 && ok) {
    mbar_arrive_expect_tx(bar_delta, (uint32_t)(cols * BM * 4));
    tma_load_2d_plain(delta_s, &tm_d, m0, tc0, bar_delta);
  }
  if (p.ks > 1) {
    cluster_sync_all();             // every CTA is past its mainloop: stage memory may be overwritten
    if (ok) {
      for (int c = h; c < p.BN / 32; c += 2) {
        const int owner = (c * 32) / cols;
        if (owner == split) continue;
        uint32_t v[32];
        tmem_ld_32x32b_x32(tmem_row + (uint32_t)(c * 32), v);
        tmem_ld_wait();
        const uint32_t base = recv + (uint32_t)(((split * cols + c * 32 - owner * cols) * BM + row) * 4);
        const uint32_t remote = map_to_cta(base, (uint32_t)owner);
#pragma unroll
        for (int i = 0; i < 32; ++i) st_cluster_f32(remote + (uint32_t)(i * BM * 4), __uint_as_float(v[i]));
      }
    }
    cluster_sync_all();             // all partials delivered
  }
  if (ok) {
    if (!mbar_wait(bar_delta, 0)) {
      flag_error(p.err, LORA_DEV_WAIT_TIMEOUT);
      ok = false;
    }
  }
  ok = __syncthreads_and(ok) != 0;
  if (ok) {
    for (int cc = h; cc < cols / 32; cc += 2) {
      const int c = split * (cols / 32) + cc;
      uint32_t v[32];
      tmem_ld_32x32b_x32(tmem_row + (uint32_t)(c * 32), v);
      tmem_ld_wait();
      if (p.ks > 1) {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          float sum = 0.f;
          for (int src = 0; src < p.ks; ++src)
            sum += src == split ? __uint_as_float(v[i])
                                : ld_shared_f32(recv + (uint32_t)(((src * cols + cc * 32 + i) * BM + row) * 4));
          v[i] = __float_as_uint(sum);
        }
      }
      const int tc = t0 + c * 32;
      const int tl = tc + lane;
      int present = 0;
      if (tl < p.T) {
        const int a = p.tok_adapter[tl];
        if (a >= 0) present = p.ptab[((int64_t)a * p.n_slots + p.slot) * kTabStride] >= 0;
      }
      const unsigned pmask = __ballot_sync(0xffffffffu, present);
      // y_s[col][feature] bf16 for the TMA store; delta_s[col][feature] fp32 from the TMA load
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const uint32_t col = (uint32_t)(cc * 32 + i);
        float acc = __uint_as_float(v[i]);
        if ((pmask >> i) & 1u) acc += ld_shared_f32(delta_s + (col * BM + row) * 4);
        st_shared_u16(y_s + (col * BM + row) * 2, f32_to_bf16_rn(acc));
      }
    }
    fence_proxy_async_shared();     // generic-proxy writes of y_s -> visible to the TMA store
  }
  __syncthreads();
  if (threadIdx.x == 0 && ok) {
    tma_store_2d(&tm_y, m0, tc0, y_s);            // rows past T and features past H are clipped
    bulk_commit_and_wait_all();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, ncols);
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

int launch_gemm(const GemmLaunch& G, cudaStream_t st) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(gemm_lora_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return lora_cuda_fail(e, "gemm_lora_kernel attribute");
    attr_set = true;
  }
  const int n_sm = device_sm_count();
  const int n_tiles = (G.T + MAX_BN - 1) / MAX_BN;
  int bn = (G.T + n_tiles - 1) / n_tiles;
  bn = ((bn + 31) / 32) * 32;
  if (bn > MAX_BN) bn = MAX_BN;
  const int m_tiles = (G.H + BM - 1) / BM;
  const int n_kb = G.H / BK;
  // Split K over a cluster while the grid would leave most SMs idle.
  int ks = 1;
  while (ks < 8 && m_tiles * n_tiles * ks * 2 <= n_sm && n_kb / (ks * 2) >= 4 && bn % (32 * ks * 2) == 0) ks *= 2;
  CUtensorMap tm_w, tm_x;
  int rc = encode_2d(&tm_w, G.W, (uint64_t)G.H, (uint64_t)G.H, BM);
  if (rc != LORA_OK) return rc;
  rc = encode_2d(&tm_x, G.x, (uint64_t)G.H, (uint64_t)G.T, (uint32_t)bn);
  if (rc != LORA_OK) return rc;
  // The delta sub-tile a CTA adds and the output sub-tile it writes: [bn/ks tokens][128 features].
  CUtensorMap tm_d, tm_y;
  rc = encode_2d_plain(&tm_d, G.delta, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, (uint64_t)G.H, (uint64_t)G.T,
                       (uint32_t)(bn / ks));
  if (rc != LORA_OK) return rc;
  rc = encode_2d_plain(&tm_y, G.y, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)G.H, (uint64_t)G.T, (uint32_t)(bn / ks));
  if (rc != LORA_OK) return rc;
  GemmParams P;
  P.y = G.y;
  P.delta = G.delta;
  P.tok_adapter = G.tok_adapter;
  P.ptab = G.ptab;
  P.err = G.err;
  P.T = G.T;
  P.H = G.H;
  P.BN = bn;
  P.n_kb = n_kb;
  P.ks = ks;
  P.slot = G.slot;
  P.n_slots = G.n_slots;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ks, m_tiles, (G.T + bn - 1) / bn);
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = st;
  cudaLaunchAttribute attrs[2];
  attrs[0].id = cudaLaunchAttributeClusterDimension;
  attrs[0].val.clusterDim.x = ks;
  attrs[0].val.clusterDim.y = 1;
  attrs[0].val.clusterDim.z = 1;
  attrs[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = G.pdl ? 2 : 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, gemm_lora_kernel, tm_w, tm_x, tm_d, tm_y, P);
  if (e == cudaSuccess) e = cudaGetLastError();
  return e == cudaSuccess ? LORA_OK : lora_cuda_fail(e, "gemm_lora_kernel launch");
}
