// Paged-gather shrink and expand: the two skinny products of the unmerged LoRA term.
//
// "S-LoRA, in depth", section "Merge or keep adapters separate": besides the shared xW,
// each token needs (xA)B for its own adapter, two skinny matmuls.  Section "Kernels for a
// batch of mixed ranks": A and B sit in scattered pool pages and ranks differ inside one
// batch, so the kernels gather pages through the page table.
//
// Both kernels walk work lists built per batch by the segment builder, so each unit
// serves a run of tokens that share one adapter and every page is fetched once per unit:
//   shrink  s[t, j]     = sum_k x[t, k] * A[k, j]   unit = (segment, 8 tokens, 8 ranks)
//   expand  delta[t, n] = sum_j s[t, j] * B[j, n]    unit = (segment, 32 tokens, 512 features)
// Page data is staged into shared memory with 1-D TMA bulk copies (cp.async.bulk, completion
// tracked by an mbarrier): a single thread keeps tens of KB per CTA in flight, which is what
// a scattered-page gather needs to approach HBM bandwidth.  bf16 inputs, fp32 accumulation,
// and a fixed summation order that depends neither on page placement nor on the other
// tokens of the batch.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "lora_internal.h"

namespace {

constexpr uint64_t kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ void flag_error(int32_t* err, int32_t bits) {
  atomicCAS(err, 0, LORA_EDEVICE);
  atomicOr(err + 1, bits);
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void bf16x8_to_f32(const uint4& v, float* f) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// ---- mbarrier + bulk copy -----------------------------------------------------------------
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
__device__ __noinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (true) {
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 > kWaitLimitNs) return false;
  }
}
// Copy `bytes` (multiple of 16, both addresses 16-byte aligned) from global to shared memory;
// completion is counted on `bar` as transaction bytes.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}
__device__ __forceinline__ void fence_barrier_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }

// ---------------------------------------------------------------------------------------
// Shrink.  8 warps, warp w <-> rank column j0 + w.  K is walked in 2048-element chunks; each
// chunk of the unit's 8 A pages and 8 x rows (up to 64 KB) is bulk-copied into one of two
// buffers while the other is being consumed.  Lanes split a chunk into 16-byte vectors; one
// warp reduction per token finishes each dot product.
// ---------------------------------------------------------------------------------------
constexpr int kShrinkThreads = 256;
constexpr int TB = kShrinkTokBlock, RG = kShrinkRankGroup;
constexpr int kShrinkChunk = 2048;                              // K elements per stage
constexpr int kShrinkRowBytes = kShrinkChunk * 2;               // 4 KB per row per stage
constexpr int kShrinkStageBytes = (RG + TB) * kShrinkRowBytes;  // 64 KB
constexpr int kShrinkSmem = 2 * kShrinkStageBytes + 128;

__global__ void __launch_bounds__(kShrinkThreads, 1)
shrink_kernel(LoraLaunch L, lora_segments seg) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int32_t sh_tok[TB];
  __shared__ int64_t sh_page[RG];
  __shared__ int32_t sh_ok;
  __shared__ __align__(8) uint64_t bars[2];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t s_base = smem_u32(smem);
  const uint32_t bar0 = smem_u32(&bars[0]);
  if (tid == 0) {
    mbar_init(bar0, 1);
    mbar_init(bar0 + 8, 1);
    fence_barrier_init();
  }
  __syncthreads();
  pdl_wait_then_release();
  const int n_work = *seg.n_shrink;
  const int H = L.H;
  const int n_kc = (H + kShrinkChunk - 1) / kShrinkChunk;
  uint32_t issued = 0, consumed = 0;   // stage counters across units (buffer = count & 1)
  bool alive = true;

  for (int w = blockIdx.x; w < n_work && alive; w += gridDim.x) {
    const int s = seg.shrink_work[4 * w], tb = seg.shrink_work[4 * w + 1], g = seg.shrink_work[4 * w + 2];
    const int a = seg.seg_adapter[s];
    const int r = L.rank[a];
    const int32_t* tab = L.ptab + ((int64_t)a * L.n_slots + L.slot) * kTabStride;   // [0][j]: A pages
    const int t_begin = seg.seg_off[s] + tb * TB;
    const int n_tok = min(TB, seg.seg_off[s + 1] - t_begin);
    const int j0 = g * RG;
    const int n_j = min(RG, r - j0);
    if (tid == 0) sh_ok = (tab[0] >= 0);      // -1: this adapter has no LoRA on this slot
    if (tid < TB) sh_tok[tid] = tid < n_tok ? seg.perm[t_begin + tid] : -1;
    if (tid >= 32 && tid < 32 + RG) {
      const int j = tid - 32;
      const bool live = j < n_j && tab[0] >= 0;
      int64_t pg = live ? tab[j0 + j] : -1;
      if (live && (pg < 0 || pg >= L.num_pages)) {
        flag_error(L.err, LORA_DEV_BAD_PAGE);
        pg = -1;
      }
      sh_page[j] = pg;
    }
    __syncthreads();
    if (!sh_ok) {
      __syncthreads();
      continue;
    }
    // One thread issues the copies of one stage: the unit's live pages and token rows.
    auto issue = [&](int kc) {
      const uint32_t buf = issued & 1;
      const int k0 = kc * kShrinkChunk;
      const uint32_t row_bytes = (uint32_t)min(kShrinkChunk, H - k0) * 2;
      uint32_t n_rows = 0;
      for (int j = 0; j < RG; ++j) n_rows += sh_page[j] >= 0;
      n_rows += n_tok;
      const uint32_t bar = bar0 + 8 * buf;
      mbar_arrive_expect_tx(bar, n_rows * row_bytes);
      const uint32_t dst = s_base + buf * kShrinkStageBytes;
      for (int j = 0; j < RG; ++j)
        if (sh_page[j] >= 0) bulk_g2s(dst + j * kShrinkRowBytes, L.pool + sh_page[j] * H + k0, row_bytes, bar);
      for (int i = 0; i < n_tok; ++i)
        bulk_g2s(dst + (RG + i) * kShrinkRowBytes, L.x + (int64_t)sh_tok[i] * H + k0, row_bytes, bar);
      ++issued;
    };
    if (tid == 0) {
      issue(0);
      if (n_kc > 1) issue(1);
    }
    float acc[TB];
#pragma unroll
    for (int i = 0; i < TB; ++i) acc[i] = 0.f;
    const bool my_page = warp < n_j && sh_page[warp] >= 0;
    for (int kc = 0; kc < n_kc; ++kc) {
      const uint32_t buf = consumed & 1;
      const uint32_t parity = (consumed >> 1) & 1;
      if (!mbar_wait(bar0 + 8 * buf, parity)) {
        if (lane == 0) flag_error(L.err, LORA_DEV_WAIT_TIMEOUT);
        alive = false;
      }
      ++consumed;
      const int k0 = kc * kShrinkChunk;
      const int n_vec = min(kShrinkChunk, H - k0) / 8;
      const uint8_t* stage = smem + buf * kShrinkStageBytes;
      if (alive && my_page) {
        const uint4* Arow = reinterpret_cast<const uint4*>(stage + warp * kShrinkRowBytes);
        for (int v = lane; v < n_vec; v += 32) {
          float af[8];
          bf16x8_to_f32(Arow[v], af);
#pragma unroll
          for (int i = 0; i < TB; ++i) {
            if (i < n_tok) {
              float xf[8];
              bf16x8_to_f32(reinterpret_cast<const uint4*>(stage + (RG + i) * kShrinkRowBytes)[v], xf);
              float d = acc[i];
#pragma unroll
              for (int e = 0; e < 8; ++e) d = fmaf(xf[e], af[e], d);
              acc[i] = d;
            }
          }
        }
      }
      alive = __syncthreads_and(alive) != 0;       // every warp is done with this buffer
      if (tid == 0 && alive && kc + 2 < n_kc) issue(kc + 2);
    }
    if (alive && my_page) {
#pragma unroll
      for (int i = 0; i < TB; ++i) {
        float v = acc[i];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0 && i < n_tok) seg.s[(int64_t)sh_tok[i] * LORA_MAX_RANK + j0 + warp] = v;
      }
    }
    __syncthreads();
  }
  // A timed-out CTA may still have copies in flight: wait (bounded) for what it issued.
  if (!alive && threadIdx.x == 0)
    while (consumed < issued) {
      (void)mbar_wait(bar0 + 8 * (consumed & 1), (consumed >> 1) & 1);
      ++consumed;
    }
}

// ---------------------------------------------------------------------------------------
// Expand.  A unit is (segment, up to 32 tokens, 512 features): the adapter's r B-page slices
// of 1 KB each are bulk-copied into shared memory at once (<= 64 KB), the tokens' s values
// (<= 8 KB) are read alongside, then 128 threads x 4 features accumulate 8 tokens at a time
// and write the fp32 delta rows.
// ---------------------------------------------------------------------------------------
constexpr int kExpandThreads = 128;
constexpr int kExpandFeat = 512;
constexpr int ETB = kExpandTokBlock;       // tokens per unit
constexpr int kExpandSmem = LORA_MAX_RANK * kExpandFeat * 2 + ETB * LORA_MAX_RANK * 4 + 128;

__global__ void __launch_bounds__(kExpandThreads)
expand_kernel(LoraLaunch L, lora_segments seg) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int64_t sh_page[LORA_MAX_RANK];
  __shared__ int32_t sh_tok[ETB];
  __shared__ int32_t sh_ok;
  __shared__ __align__(8) uint64_t bar_s;
  const int tid = threadIdx.x;
  uint16_t* Bs = reinterpret_cast<uint16_t*>(smem);                                  // [64][512]
  float* S = reinterpret_cast<float*>(smem + LORA_MAX_RANK * kExpandFeat * 2);       // [ETB][64]
  const uint32_t bar = smem_u32(&bar_s);
  if (tid == 0) {
    mbar_init(bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  pdl_wait_then_release();
  const int H = L.H;
  const int n_fc = (H + kExpandFeat - 1) / kExpandFeat;
  const int n_units = *seg.n_expand * n_fc;
  uint32_t phase = 0;

  for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
    const int w = u / n_fc, fc = u % n_fc;
    const int s = seg.expand_work[2 * w], tg = seg.expand_work[2 * w + 1];
    const int a = seg.seg_adapter[s];
    const int r = L.rank[a];
    const int32_t* tab = L.ptab + ((int64_t)a * L.n_slots + L.slot) * kTabStride + LORA_MAX_RANK;  // B pages
    const int t_begin = seg.seg_off[s] + tg * ETB;
    const int n_tok = min(ETB, seg.seg_off[s + 1] - t_begin);
    const int f0 = fc * kExpandFeat;
    const int nf = min(kExpandFeat, H - f0);
    if (tid == 0) sh_ok = (tab[0] >= 0);
    if (tid < ETB) sh_tok[tid] = tid < n_tok ? seg.perm[t_begin + tid] : -1;
    if (tid < LORA_MAX_RANK) {
      const bool live = tid < r && tab[0] >= 0;
      int64_t pg = live ? tab[tid] : -1;
      if (live && (pg < 0 || pg >= L.num_pages)) {
        flag_error(L.err, LORA_DEV_BAD_PAGE);
        pg = -1;
      }
      sh_page[tid] = pg;
    }
    __syncthreads();
    if (!sh_ok) {
      __syncthreads();
      continue;
    }
    if (tid == 0) {
      uint32_t n_live = 0;
      for (int j = 0; j < r; ++j) n_live += sh_page[j] >= 0;
      mbar_arrive_expect_tx(bar, n_live * (uint32_t)nf * 2);
      for (int j = 0; j < r; ++j)
        if (sh_page[j] >= 0) bulk_g2s(smem_u32(Bs + j * kExpandFeat), L.pool + sh_page[j] * H + f0, (uint32_t)nf * 2, bar);
    }
    // s values of the unit's tokens (zero for missing pages and tokens), alongside the copies
    for (int i = tid; i < ETB * LORA_MAX_RANK; i += kExpandThreads) {
      const int tk = i / LORA_MAX_RANK, j = i % LORA_MAX_RANK;
      S[i] = (tk < n_tok && j < r && sh_page[j] >= 0) ? seg.s[(int64_t)sh_tok[tk] * LORA_MAX_RANK + j] : 0.f;
    }
    bool ok = mbar_wait(bar, phase);
    phase ^= 1;
    if (!ok) flag_error(L.err, LORA_DEV_WAIT_TIMEOUT);
    ok = __syncthreads_and(ok) != 0;
    const int f = tid * 4;
    if (ok && f < nf) {
      for (int t8 = 0; t8 < n_tok; t8 += 8) {
        float acc[8][4];
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[i][e] = 0.f;
        for (int j = 0; j < r; ++j) {
          if (sh_page[j] < 0) continue;
          const uint2 bv = *reinterpret_cast<const uint2*>(Bs + j * kExpandFeat + f);
          const float b[4] = {__uint_as_float(bv.x << 16), __uint_as_float(bv.x & 0xFFFF0000u),
                              __uint_as_float(bv.y << 16), __uint_as_float(bv.y & 0xFFFF0000u)};
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float sv = S[(t8 + i) * LORA_MAX_RANK + j];
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[i][e] = fmaf(sv, b[e], acc[i][e]);
          }
        }
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (t8 + i < n_tok)
            *reinterpret_cast<float4*>(L.delta + (int64_t)sh_tok[t8 + i] * H + f0 + f) =
                make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
      }
    }
    __syncthreads();                                  // buffers are reused by the next unit
    if (!ok) break;
  }
}

inline int grid_cap(int upper, int cap) { return upper < cap ? (upper > 0 ? upper : 1) : cap; }

}  // namespace

// Grids loop over the work list (its length is only known on the device), capped at what
// stays resident: shrink one CTA per SM (128 KB of stages), expand three per SM.
int launch_shrink(const LoraLaunch& L, cudaStream_t st) {
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(shrink_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kShrinkSmem);
    if (e != cudaSuccess) return lora_cuda_fail(e, "shrink_kernel attribute");
    attr = true;
  }
  const int grid = grid_cap(L.seg->shrink_cap, device_sm_count());
  cudaError_t e = launch_pdl(L.pdl, shrink_kernel, dim3(grid), dim3(kShrinkThreads), kShrinkSmem, st, L, *L.seg);
  if (e == cudaSuccess) e = cudaGetLastError();
  return e == cudaSuccess ? LORA_OK : lora_cuda_fail(e, "shrink_kernel launch");
}

int launch_expand(const LoraLaunch& L, cudaStream_t st) {
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(expand_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kExpandSmem);
    if (e != cudaSuccess) return lora_cuda_fail(e, "expand_kernel attribute");
    attr = true;
  }
  const int n_fc = (L.H + kExpandFeat - 1) / kExpandFeat;
  const int grid = grid_cap(L.seg->expand_cap * n_fc, device_sm_count() * 3);
  cudaError_t e = launch_pdl(L.pdl, expand_kernel, dim3(grid), dim3(kExpandThreads), kExpandSmem, st, L, *L.seg);
  if (e == cudaSuccess) e = cudaGetLastError();
  return e == cudaSuccess ? LORA_OK : lora_cuda_fail(e, "expand_kernel launch");
}
