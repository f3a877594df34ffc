// Segment builder: group a batch's tokens by adapter id, stably.
//
// The pages batch requests of many adapters into one base projection and gather each
// request's own A and B pages ("S-LoRA, in depth", section "The architecture"); grouping
// tokens by adapter lets each adapter's pages be read once per batch instead of once per
// token.  Output order: ascending adapter id, ties by token index; tokens without an
// adapter (-1) first and outside every segment.
//
// One CTA of 1024 threads: a shared-memory histogram over adapter ids, a block scan that
// turns counts into run starts and lists the non-empty adapters, then a stable scatter in
// chunks of 1024 tokens (warp-level match for ranks inside a warp, warps in order), and
// finally the work lists of the shrink and expand kernels.
#include <cuda_runtime.h>

#include "lora_internal.h"

namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;

__device__ __forceinline__ void flag_error(int32_t* err, int32_t bits) {
  atomicCAS(err, 0, LORA_EDEVICE);
  atomicOr(err + 1, bits);
}

// Exclusive block scan of two int32 values per thread; returns the totals in *tot0/*tot1.
__device__ __forceinline__ void block_exclusive_scan2(int32_t& a, int32_t& b, int32_t* sh_a, int32_t* sh_b,
                                                      int32_t* tot_a, int32_t* tot_b) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int32_t ia = a, ib = b;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int32_t va = __shfl_up_sync(0xffffffffu, ia, o);
    int32_t vb = __shfl_up_sync(0xffffffffu, ib, o);
    if (lane >= o) { ia += va; ib += vb; }
  }
  if (lane == 31) { sh_a[warp] = ia; sh_b[warp] = ib; }
  __syncthreads();
  if (warp == 0) {
    int32_t wa = sh_a[lane], wb = sh_b[lane];
    int32_t sa = wa, sb = wb;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int32_t va = __shfl_up_sync(0xffffffffu, sa, o);
      int32_t vb = __shfl_up_sync(0xffffffffu, sb, o);
      if (lane >= o) { sa += va; sb += vb; }
    }
    sh_a[lane] = sa - wa;   // exclusive prefix of warp totals
    sh_b[lane] = sb - wb;
    if (lane == 31) { sh_a[32] = sa; sh_b[32] = sb; }
  }
  __syncthreads();
  const int32_t ea = sh_a[warp] + ia - a, eb = sh_b[warp] + ib - b;
  *tot_a = sh_a[32];
  *tot_b = sh_b[32];
  a = ea;
  b = eb;
  __syncthreads();
}

__global__ void __launch_bounds__(kThreads, 1)
segments_kernel(const int32_t* __restrict__ token_adapter, int32_t T, const int32_t* __restrict__ rank,
                int32_t max_adapters, lora_segments seg, int32_t* __restrict__ err) {
  extern __shared__ int32_t cnt[];           // [max_adapters + 1], key = adapter id + 1 (0 = none)
  __shared__ int32_t sh_a[33], sh_b[33];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int K = max_adapters + 1;
  pdl_wait_then_release();

  for (int k = tid; k < K; k += kThreads) cnt[k] = 0;
  __syncthreads();

  // 1. validate ids and count tokens per key
  for (int t = tid; t < T; t += kThreads) {
    const int32_t a = token_adapter[t];
    int32_t key = 0;
    if (a >= 0 && a < max_adapters && rank[a] > 0) {
      key = a + 1;
    } else if (a != -1) {
      flag_error(err, LORA_DEV_UNKNOWN_ADAPTER);
    }
    seg.tok_adapter[t] = key - 1;
    atomicAdd(&cnt[key], 1);
  }
  __syncthreads();

  // 2. run starts per key, list of non-empty adapters (the segments)
  const int per = (K + kThreads - 1) / kThreads;
  const int k_lo = min(K, tid * per), k_hi = min(K, k_lo + per);
  int32_t csum = 0, nz = 0;
  for (int k = k_lo; k < k_hi; ++k) {
    csum += cnt[k];
    nz += (k > 0 && cnt[k] > 0);
  }
  int32_t tot_c, tot_nz;
  block_exclusive_scan2(csum, nz, sh_a, sh_b, &tot_c, &tot_nz);
  for (int k = k_lo; k < k_hi; ++k) {
    const int32_t c = cnt[k];
    if (k > 0 && c > 0) {
      seg.seg_off[nz] = csum;
      seg.seg_adapter[nz] = k - 1;
      ++nz;
    }
    cnt[k] = csum;      // becomes the running write position of key k
    csum += c;
  }
  const int32_t S = tot_nz;
  if (tid == 0) {
    seg.seg_off[S] = T;
    if (S == 0) seg.seg_off[0] = T;
    *seg.n_seg = S;
  }
  __syncthreads();

  // 3. stable scatter, 1024 tokens at a time; warps take their turn in index order
  for (int base_t = 0; base_t < T; base_t += kThreads) {
    const int t = base_t + tid;
    const bool valid = t < T;
    const int32_t key = valid ? seg.tok_adapter[t] + 1 : -1;
    const unsigned peers = __match_any_sync(0xffffffffu, key);
    const int lrank = __popc(peers & ((1u << lane) - 1u));
    const int leader = __ffs(peers) - 1;
    for (int w = 0; w < kWarps; ++w) {
      if (warp == w) {
        int32_t pos = 0;
        if (valid && lane == leader) {
          pos = cnt[key];
          cnt[key] = pos + __popc(peers);
        }
        pos = __shfl_sync(0xffffffffu, pos, leader);
        if (valid) seg.perm[pos + lrank] = t;
      }
      __syncthreads();
    }
  }

  // 4. work lists: expand units (segment, token block); shrink units (segment, token block, rank group)
  const int sper = (S + kThreads - 1) / kThreads;
  const int s_lo = min(S, tid * sper), s_hi = min(S, s_lo + sper);
  int32_t ne = 0, ns = 0;
  for (int s = s_lo; s < s_hi; ++s) {
    const int32_t n = seg.seg_off[s + 1] - seg.seg_off[s];
    const int32_t r = rank[seg.seg_adapter[s]];
    ne += (n + kExpandTokBlock - 1) / kExpandTokBlock;
    ns += ((n + kShrinkTokBlock - 1) / kShrinkTokBlock) * ((r + kShrinkRankGroup - 1) / kShrinkRankGroup);
  }
  int32_t tot_e, tot_s;
  block_exclusive_scan2(ne, ns, sh_a, sh_b, &tot_e, &tot_s);
  for (int s = s_lo; s < s_hi; ++s) {
    const int32_t n = seg.seg_off[s + 1] - seg.seg_off[s];
    const int32_t r = rank[seg.seg_adapter[s]];
    const int32_t nbe = (n + kExpandTokBlock - 1) / kExpandTokBlock;
    for (int b = 0; b < nbe; ++b, ++ne) {
      seg.expand_work[2 * ne] = s;
      seg.expand_work[2 * ne + 1] = b;
    }
    const int32_t nbs = (n + kShrinkTokBlock - 1) / kShrinkTokBlock;
    const int32_t ng = (r + kShrinkRankGroup - 1) / kShrinkRankGroup;
    for (int b = 0; b < nbs; ++b)
      for (int g = 0; g < ng; ++g, ++ns) {
        seg.shrink_work[4 * ns] = s;
        seg.shrink_work[4 * ns + 1] = b;
        seg.shrink_work[4 * ns + 2] = g;
        seg.shrink_work[4 * ns + 3] = 0;
      }
  }
  if (tid == 0) {
    *seg.n_expand = tot_e;
    *seg.n_shrink = tot_s;
  }
}

}  // namespace

int launch_segments_build(const lora_pool* p, const int32_t* token_adapter, int32_t T, const lora_segments* seg,
                          cudaStream_t st, bool pdl) {
  const size_t smem = (size_t)(p->max_adapters + 1) * sizeof(int32_t);
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(segments_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)((LORA_MAX_ADAPTERS + 1) * sizeof(int32_t)));
    if (e != cudaSuccess) return lora_cuda_fail(e, "segments_kernel attribute");
    attr_set = true;
  }
  cudaError_t e = launch_pdl(pdl, segments_kernel, dim3(1), dim3(kThreads), smem, st, token_adapter, T,
                             (const int32_t*)p->d_rank, p->max_adapters, *seg, p->d_err);
  if (e == cudaSuccess) e = cudaGetLastError();
  return e == cudaSuccess ? LORA_OK : lora_cuda_fail(e, "segments_kernel launch");
}

extern "C" int lora_segments_build(lora_pool* p, const int32_t* token_adapter, int32_t T, lora_segments* seg,
                                   lora_stream_t stream) {
  if (!p || !seg || T < 0 || (T > 0 && !token_adapter)) return lora_fail(LORA_EINVAL, "lora_segments_build: bad arguments");
  if (p->planning) return lora_fail(LORA_EINVAL, "lora_segments_build: planning pool has no device state");
  if (T > seg->T_max) return lora_fail(LORA_EINVAL, "lora_segments_build: T exceeds the workspace's T_max");
  if (seg->H != p->H) return lora_fail(LORA_EINVAL, "lora_segments_build: workspace was sized for another pool");
  int rc;
  {
    ProfScope prof(p, LORA_KIND_SEGMENTS, reinterpret_cast<cudaStream_t>(stream));
    rc = launch_segments_build(p, token_adapter, T, seg, reinterpret_cast<cudaStream_t>(stream), !p->prof_on);
  }
  if (rc == LORA_OK) seg->T = T;
  return rc;
}
