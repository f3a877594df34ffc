// Paged-gather shrink and expand: the two skinny products of the unmerged LoRA term.
//
// "S-LoRA, in depth", section "Merge or keep adapters separate": besides the shared xW,
// each token needs (xA)B for its own adapter, two skinny matmuls.  Section "Kernels for a
// batch of mixed ranks": A and B sit in scattered pool pages and ranks differ inside one
// batch, so the kernels gather pages through the page table.
//
// Both kernels walk work lists built per batch by the segment builder, so each unit
// serves a run of tokens that share one adapter and every page is read once per unit:
//   shrink  s[t, j]     = sum_k x[t, k] * A[k, j]            unit = (segment, 8 tokens, 8 ranks)
//   expand  delta[t, n] = sum_j s[t, j] * B[j, n]             unit = (segment, 8 tokens) x 2048 features
// bf16 inputs, fp32 accumulation, fixed summation order (independent of page placement and
// of the rest of the batch).  Page loads are 16-byte vectors, coalesced along the page.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "lora_internal.h"

namespace {

__device__ __forceinline__ void flag_error(int32_t* err, int32_t bits) {
  atomicCAS(err, 0, LORA_EDEVICE);
  atomicOr(err + 1, bits);
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4& v, float* f) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ uint4 ldg16(const void* p) { return __ldg(reinterpret_cast<const uint4*>(p)); }

// ---------------------------------------------------------------------------------------
// Shrink.  128 threads split H in 16-byte chunks; each thread keeps 8 tokens x 8 ranks of
// partial dot products; a warp butterfly reduce-scatter plus a 4-warp shared-memory sum
// finishes them.
// ---------------------------------------------------------------------------------------
constexpr int kShrinkThreads = 128;
constexpr int TB = kShrinkTokBlock, RG = kShrinkRankGroup;

__global__ void __launch_bounds__(kShrinkThreads)
shrink_kernel(LoraLaunch L, lora_segments seg) {
  __shared__ int32_t sh_tok[TB];
  __shared__ int64_t sh_page[RG];
  __shared__ int32_t sh_ok;
  __shared__ float sh_red[kShrinkThreads / 32][TB * RG];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n_work = *seg.n_shrink;
  const int H = L.H;
  const int n_chunks = H / 8;

  for (int w = blockIdx.x; w < n_work; w += gridDim.x) {
    const int s = seg.shrink_work[4 * w], tb = seg.shrink_work[4 * w + 1], g = seg.shrink_work[4 * w + 2];
    const int a = seg.seg_adapter[s];
    const int r = L.rank[a];
    const int32_t* tab = L.ptab + ((int64_t)a * L.n_slots + L.slot) * kTabStride;   // [0][j]: A pages
    const int t_begin = seg.seg_off[s] + tb * TB;
    const int n_tok = min(TB, seg.seg_off[s + 1] - t_begin);
    const int j0 = g * RG;
    const int n_j = min(RG, r - j0);
    if (tid == 0) sh_ok = (tab[0] >= 0);      // -1: this adapter has no LoRA on this slot
    if (tid < TB) sh_tok[tid] = tid < n_tok ? seg.perm[t_begin + tid] : 0;
    if (tid >= 32 && tid < 32 + RG) {
      const int j = tid - 32;
      const bool live = j < n_j && tab[0] >= 0;   // a slot without LoRA has only -1 entries
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

    float acc[TB][RG];
#pragma unroll
    for (int i = 0; i < TB; ++i)
#pragma unroll
      for (int j = 0; j < RG; ++j) acc[i][j] = 0.f;

    for (int c = tid; c < n_chunks; c += kShrinkThreads) {
      float af[RG][8];
#pragma unroll
      for (int j = 0; j < RG; ++j) {
        const int64_t pg = sh_page[j];
        uint4 v = make_uint4(0, 0, 0, 0);
        if (pg >= 0) v = ldg16(L.pool + pg * H + (int64_t)c * 8);
        bf16x8_to_f32(v, af[j]);
      }
#pragma unroll
      for (int i = 0; i < TB; ++i) {
        if (i < n_tok) {
          float xf[8];
          bf16x8_to_f32(ldg16(L.x + (int64_t)sh_tok[i] * H + (int64_t)c * 8), xf);
#pragma unroll
          for (int j = 0; j < RG; ++j) {
            float d = acc[i][j];
#pragma unroll
            for (int e = 0; e < 8; ++e) d = fmaf(xf[e], af[j][e], d);
            acc[i][j] = d;
          }
        }
      }
    }

    // Butterfly reduce-scatter of 64 values over the warp: lane ends with entries 2*lane, 2*lane+1.
    float* v = &acc[0][0];
#pragma unroll
    for (int m = TB * RG; m >= 4; m >>= 1) {   // m live values -> m/2
      const int off = m / 4;                     // lane bit that picks the half a lane keeps
      const bool upper = (lane & off) != 0;
#pragma unroll
      for (int i = 0; i < m / 2; ++i) {
        const float keep = upper ? v[m / 2 + i] : v[i];
        const float send = upper ? v[i] : v[m / 2 + i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
      }
    }
    sh_red[warp][2 * lane] = v[0];
    sh_red[warp][2 * lane + 1] = v[1];
    __syncthreads();
    if (tid < TB * RG) {
      const int i = tid / RG, j = tid % RG;
      float sum = 0.f;
#pragma unroll
      for (int q = 0; q < kShrinkThreads / 32; ++q) sum += sh_red[q][tid];
      if (i < n_tok && j < n_j) seg.s[(int64_t)sh_tok[i] * LORA_MAX_RANK + j0 + j] = sum;
    }
    __syncthreads();
  }
}

// ---------------------------------------------------------------------------------------
// Expand.  256 threads x 8 features = 2048 features per CTA (grid.y covers H); each thread
// streams its 16-byte slice of the adapter's r B pages and keeps 8 tokens x 8 features.
// ---------------------------------------------------------------------------------------
constexpr int kExpandThreads = 256;
constexpr int kExpandFeat = kExpandThreads * 8;
constexpr int ETB = kExpandTokBlock;

__global__ void __launch_bounds__(kExpandThreads)
expand_kernel(LoraLaunch L, lora_segments seg) {
  __shared__ float sh_s[ETB][LORA_MAX_RANK];
  __shared__ int64_t sh_page[LORA_MAX_RANK];
  __shared__ int32_t sh_tok[ETB];
  __shared__ int32_t sh_ok;
  const int tid = threadIdx.x;
  const int n_work = *seg.n_expand;
  const int H = L.H;
  const int f = blockIdx.y * kExpandFeat + tid * 8;

  for (int w = blockIdx.x; w < n_work; w += gridDim.x) {
    const int s = seg.expand_work[2 * w], tb = seg.expand_work[2 * w + 1];
    const int a = seg.seg_adapter[s];
    const int r = L.rank[a];
    const int32_t* tab = L.ptab + ((int64_t)a * L.n_slots + L.slot) * kTabStride + LORA_MAX_RANK;  // B pages
    const int t_begin = seg.seg_off[s] + tb * ETB;
    const int n_tok = min(ETB, seg.seg_off[s + 1] - t_begin);
    if (tid == 0) sh_ok = (tab[0] >= 0);
    if (tid < ETB) sh_tok[tid] = tid < n_tok ? seg.perm[t_begin + tid] : 0;
    if (tid < LORA_MAX_RANK) {
      const bool live = tid < r && tab[0] >= 0;   // a slot without LoRA has only -1 entries
      int64_t pg = live ? tab[tid] : -1;
      if (live && (pg < 0 || pg >= L.num_pages)) {
        flag_error(L.err, LORA_DEV_BAD_PAGE);
        pg = -1;
      }
      sh_page[tid] = pg;
    }
    __syncthreads();
    for (int i = tid; i < ETB * LORA_MAX_RANK; i += kExpandThreads) {
      const int tk = i / LORA_MAX_RANK, j = i % LORA_MAX_RANK;
      sh_s[tk][j] = (tk < n_tok && j < r) ? seg.s[(int64_t)sh_tok[tk] * LORA_MAX_RANK + j] : 0.f;
    }
    __syncthreads();
    if (sh_ok && f < H) {
      float acc[ETB][8];
#pragma unroll
      for (int i = 0; i < ETB; ++i)
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[i][e] = 0.f;
      int j = 0;
      for (; j + 4 <= r; j += 4) {
        uint4 bv[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int64_t pg = sh_page[j + u];
          bv[u] = pg >= 0 ? ldg16(L.pool + pg * H + f) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          float bf[8];
          bf16x8_to_f32(bv[u], bf);
#pragma unroll
          for (int i = 0; i < ETB; ++i) {
            const float sv = sh_s[i][j + u];
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[i][e] = fmaf(sv, bf[e], acc[i][e]);
          }
        }
      }
      for (; j < r; ++j) {
        const int64_t pg = sh_page[j];
        float bf[8];
        bf16x8_to_f32(pg >= 0 ? ldg16(L.pool + pg * H + f) : make_uint4(0, 0, 0, 0), bf);
#pragma unroll
        for (int i = 0; i < ETB; ++i) {
          const float sv = sh_s[i][j];
#pragma unroll
          for (int e = 0; e < 8; ++e) acc[i][e] = fmaf(sv, bf[e], acc[i][e]);
        }
      }
#pragma unroll
      for (int i = 0; i < ETB; ++i) {
        if (i < n_tok) {
          float4* dst = reinterpret_cast<float4*>(L.delta + (int64_t)sh_tok[i] * H + f);
          dst[0] = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
          dst[1] = make_float4(acc[i][4], acc[i][5], acc[i][6], acc[i][7]);
        }
      }
    }
    __syncthreads();
  }
}

inline int grid_cap(int upper, int cap) { return upper < cap ? (upper > 0 ? upper : 1) : cap; }

}  // namespace

int launch_shrink(const LoraLaunch& L, cudaStream_t st) {
  const int grid = grid_cap(L.seg->shrink_cap, 152 * 16);
  shrink_kernel<<<grid, kShrinkThreads, 0, st>>>(L, *L.seg);
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? LORA_OK : lora_cuda_fail(e, "shrink_kernel launch");
}

int launch_expand(const LoraLaunch& L, cudaStream_t st) {
  const dim3 grid(grid_cap(L.seg->expand_cap, 152 * 8), (L.H + kExpandFeat - 1) / kExpandFeat);
  expand_kernel<<<grid, kExpandThreads, 0, st>>>(L, *L.seg);
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? LORA_OK : lora_cuda_fail(e, "expand_kernel launch");
}
