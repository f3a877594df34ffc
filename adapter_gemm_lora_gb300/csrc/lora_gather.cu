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
//   expand  delta[t, n] = sum_j s[t, j] * B[j, n]    unit = (segment, 32 tokens, 1024 features)
// A page gather is latency-bound unless many bytes are in flight: every lane issues 8 to 16
// independent 16-byte loads before using any of them, and no barrier sits inside a unit, so
// all resident warps keep the memory system busy.  bf16 inputs, fp32 accumulation, and a
// fixed summation order that depends neither on page placement nor on the other tokens of
// the batch.
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
// Shrink.  A unit is (segment, up to 8 tokens, 8 rank columns); warp w computes column j0 + w:
// its A page streams through registers in rounds of 8 x 16-byte loads per lane (4 KB per warp
// in flight), each token row of the unit is read at the same positions, and one warp
// reduction per token finishes each dot product.  No shared-memory staging and no barrier
// inside a unit, so every resident warp keeps loads in flight.
// ---------------------------------------------------------------------------------------
constexpr int kShrinkThreads = 256;
constexpr int TB = kShrinkTokBlock, RG = kShrinkRankGroup;
constexpr int kShrinkRound = 8;                 // 16-byte vectors per lane per round

__device__ __forceinline__ float dot8(const uint4& a, const uint4& b, float acc) {
  float af[8], bf[8];
  bf16x8_to_f32(a, af);
  bf16x8_to_f32(b, bf);
#pragma unroll
  for (int e = 0; e < 8; ++e) acc = fmaf(af[e], bf[e], acc);
  return acc;
}

__global__ void __launch_bounds__(kShrinkThreads, 2)
shrink_kernel(LoraLaunch L, lora_segments seg) {
  __shared__ int32_t sh_tok[TB];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  pdl_wait_then_release();
  const int n_work = *seg.n_shrink;
  const int H = L.H;
  const int n_vec = H / 8;                      // 16-byte vectors per page

  for (int w = blockIdx.x; w < n_work; w += gridDim.x) {
    const int s = seg.shrink_work[4 * w], tb = seg.shrink_work[4 * w + 1], g = seg.shrink_work[4 * w + 2];
    const int a = seg.seg_adapter[s];
    const int r = L.rank[a];
    const int32_t* tab = L.ptab + ((int64_t)a * L.n_slots + L.slot) * kTabStride;   // [0][j]: A pages
    const int t_begin = seg.seg_off[s] + tb * TB;
    const int n_tok = min(TB, seg.seg_off[s + 1] - t_begin);
    const int j = g * RG + warp;
    __syncthreads();                            // previous unit done with sh_tok
    if (tid < TB) sh_tok[tid] = tid < n_tok ? seg.perm[t_begin + tid] : 0;
    __syncthreads();
    if (tab[0] < 0 || j >= r) continue;         // no LoRA on this slot / column beyond the rank
    const int64_t pg = tab[j];
    if (pg < 0 || pg >= L.num_pages) {
      if (lane == 0) flag_error(L.err, LORA_DEV_BAD_PAGE);
      continue;
    }
    const uint4* A = reinterpret_cast<const uint4*>(L.pool + pg * H);
    float acc[TB];
#pragma unroll
    for (int i = 0; i < TB; ++i) acc[i] = 0.f;
    // Per round: the A vectors and the first token's row are loaded together; while a token's
    // row is being multiplied, the next token's row is already in flight.
    for (int base = 0; base < n_vec; base += 32 * kShrinkRound) {
      uint4 av[kShrinkRound], xa[kShrinkRound], xb[kShrinkRound];
#pragma unroll
      for (int u = 0; u < kShrinkRound; ++u) {
        const int v = base + u * 32 + lane;
        av[u] = v < n_vec ? __ldg(A + v) : make_uint4(0, 0, 0, 0);
        xa[u] = v < n_vec ? __ldg(reinterpret_cast<const uint4*>(L.x + (int64_t)sh_tok[0] * H) + v)
                          : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int i = 0; i < TB; i += 2) {
        if (i + 1 < n_tok) {
#pragma unroll
          for (int u = 0; u < kShrinkRound; ++u) {
            const int v = base + u * 32 + lane;
            xb[u] = v < n_vec ? __ldg(reinterpret_cast<const uint4*>(L.x + (int64_t)sh_tok[i + 1] * H) + v)
                              : make_uint4(0, 0, 0, 0);
          }
        }
        if (i < n_tok) {
          float d = acc[i];
#pragma unroll
          for (int u = 0; u < kShrinkRound; ++u) d = dot8(av[u], xa[u], d);
          acc[i] = d;
        }
        if (i + 2 < n_tok) {
#pragma unroll
          for (int u = 0; u < kShrinkRound; ++u) {
            const int v = base + u * 32 + lane;
            xa[u] = v < n_vec ? __ldg(reinterpret_cast<const uint4*>(L.x + (int64_t)sh_tok[i + 2] * H) + v)
                              : make_uint4(0, 0, 0, 0);
          }
        }
        if (i + 1 < n_tok) {
          float d = acc[i + 1];
#pragma unroll
          for (int u = 0; u < kShrinkRound; ++u) d = dot8(av[u], xb[u], d);
          acc[i + 1] = d;
        }
      }
    }
#pragma unroll
    for (int i = 0; i < TB; ++i) {
      if (i < n_tok) {
        float v = acc[i];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) seg.s[(int64_t)sh_tok[i] * LORA_MAX_RANK + j] = v;
      }
    }
  }
}

// ---------------------------------------------------------------------------------------
// Expand.  A unit is (segment, up to 8 tokens, 1024 features); warp w owns 256 features, 8
// per lane (one 16-byte slice of each B page).  Pages are read 8 at a time (8 loads per lane
// in flight) and each slice is applied to all of the unit's tokens in the same pass, from
// their s values in shared memory; the fp32 delta rows are written with 16-byte stores.
// ---------------------------------------------------------------------------------------
constexpr int kExpandThreads = 128;
constexpr int kExpandFeat = 1024;
constexpr int ETB = kExpandTokBlock;            // tokens per unit (8)
constexpr int kExpandPages = 8;                 // pages in flight per lane

__global__ void __launch_bounds__(kExpandThreads, 4)
expand_kernel(LoraLaunch L, lora_segments seg) {
  __shared__ float S[ETB][LORA_MAX_RANK];
  __shared__ int64_t sh_page[LORA_MAX_RANK];
  __shared__ int32_t sh_tok[ETB];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  pdl_wait_then_release();
  const int H = L.H;
  const int n_fc = (H + kExpandFeat - 1) / kExpandFeat;
  const int n_units = *seg.n_expand * n_fc;

  for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
    const int w = u / n_fc, fc = u % n_fc;
    const int s = seg.expand_work[2 * w], tg = seg.expand_work[2 * w + 1];
    const int a = seg.seg_adapter[s];
    const int r = L.rank[a];
    const int32_t* tab = L.ptab + ((int64_t)a * L.n_slots + L.slot) * kTabStride + LORA_MAX_RANK;  // B pages
    const int t_begin = seg.seg_off[s] + tg * ETB;
    const int n_tok = min(ETB, seg.seg_off[s + 1] - t_begin);
    __syncthreads();                            // previous unit done with the shared arrays
    if (tab[0] < 0) continue;                   // no LoRA on this slot (uniform across the CTA)
    if (tid < ETB) sh_tok[tid] = tid < n_tok ? seg.perm[t_begin + tid] : 0;
    if (tid < LORA_MAX_RANK) {
      int64_t pg = tid < r ? tab[tid] : -1;
      if (tid < r && (pg < 0 || pg >= L.num_pages)) {
        flag_error(L.err, LORA_DEV_BAD_PAGE);
        pg = -1;
      }
      sh_page[tid] = pg;
    }
    __syncthreads();
    for (int i = tid; i < ETB * LORA_MAX_RANK; i += kExpandThreads) {
      const int tk = i / LORA_MAX_RANK, j = i % LORA_MAX_RANK;
      S[tk][j] = (tk < n_tok && j < r && sh_page[j] >= 0) ? seg.s[(int64_t)sh_tok[tk] * LORA_MAX_RANK + j] : 0.f;
    }
    __syncthreads();
    const int f = fc * kExpandFeat + warp * 256 + lane * 8;
    if (f >= H) continue;
    {
      constexpr int t0 = 0;
      float acc[ETB][8];
#pragma unroll
      for (int i = 0; i < ETB; ++i)
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[i][e] = 0.f;
      for (int j0 = 0; j0 < r; j0 += kExpandPages) {
        uint4 bv[kExpandPages];
#pragma unroll
        for (int q = 0; q < kExpandPages; ++q) {
          const int j = j0 + q;
          const int64_t pg = j < r ? sh_page[j] : -1;
          bv[q] = pg >= 0 ? __ldg(reinterpret_cast<const uint4*>(L.pool + pg * H + f)) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int q = 0; q < kExpandPages; ++q) {
          float bf[8];
          bf16x8_to_f32(bv[q], bf);
          const int j = min(j0 + q, LORA_MAX_RANK - 1);   // S is zero past the rank
#pragma unroll
          for (int i = 0; i < ETB; ++i) {
            const float sv = S[i][j];                    // zero for tokens past n_tok
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[i][e] = fmaf(sv, bf[e], acc[i][e]);
          }
        }
      }
#pragma unroll
      for (int i = 0; i < ETB; ++i) {
        if (t0 + i < n_tok) {
          float4* dst = reinterpret_cast<float4*>(L.delta + (int64_t)sh_tok[t0 + i] * H + f);
          dst[0] = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
          dst[1] = make_float4(acc[i][4], acc[i][5], acc[i][6], acc[i][7]);
        }
      }
    }
  }
}

inline int grid_cap(int upper, int cap) { return upper < cap ? (upper > 0 ? upper : 1) : cap; }

}  // namespace

// Grids loop over the work list (its length is only known on the device), capped at what
// stays resident: two shrink CTAs (8 warps each) and four expand CTAs (4 warps each) per SM.
int launch_shrink(const LoraLaunch& L, cudaStream_t st) {
  const int grid = grid_cap(L.seg->shrink_cap, device_sm_count() * 2);
  cudaError_t e = launch_pdl(L.pdl, shrink_kernel, dim3(grid), dim3(kShrinkThreads), 0, st, L, *L.seg);
  if (e == cudaSuccess) e = cudaGetLastError();
  return e == cudaSuccess ? LORA_OK : lora_cuda_fail(e, "shrink_kernel launch");
}

int launch_expand(const LoraLaunch& L, cudaStream_t st) {
  const int n_fc = (L.H + kExpandFeat - 1) / kExpandFeat;
  const int grid = grid_cap(L.seg->expand_cap * n_fc, device_sm_count() * 4);
  cudaError_t e = launch_pdl(L.pdl, expand_kernel, dim3(grid), dim3(kExpandThreads), 0, st, L, *L.seg);
  if (e == cudaSuccess) e = cudaGetLastError();
  return e == cudaSuccess ? LORA_OK : lora_cuda_fail(e, "expand_kernel launch");
}
