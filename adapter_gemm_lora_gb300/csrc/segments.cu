// Segment builder: group a batch's tokens by adapter id, stably.
//
// The pages batch requests of many adapters into one base projection and gather each
// request's own A and B pages ("S-LoRA, in depth", section "The architecture"); grouping
// tokens by adapter lets each adapter's pages be read once per batch instead of once per
// token.  Output order: ascending adapter id, ties by token index; tokens without an
// adapter (-1) first and outside every segment.
//
// One CTA of 1024 threads: a shared-memory histogram over adapter ids (with each used
// adapter's rank), two block scans that turn counts into run starts, segment indices and the
// offsets of the LoRA-delta work units within their rank class (each unit written right away
// as a complete record: adapter, rank, first index into perm, token count), then a stable
// scatter in chunks of 1024 tokens (warp-level match for ranks inside a warp, warps in order).
#include <cuda_runtime.h>

#include "lora_internal.h"

namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;

__device__ __forceinline__ void flag_error(int32_t* err, int32_t bits) {
  atomicCAS(err, 0, LORA_EDEVICE);
  atomicOr(err + 1, bits);
}

// Work-unit cost class of a rank: 0 for 33..64, 1 for 17..32, 2 for 9..16, 3 for 1..8.
__device__ __forceinline__ int rank_class(int32_t r) { return r > 32 ? 0 : r > 16 ? 1 : r > 8 ? 2 : 3; }

// Exclusive block scan of four int32 values per thread; totals land in tot[0..3].
__device__ __forceinline__ void block_exclusive_scan4(int32_t (&v)[4], int32_t (*sh)[33], int32_t (&tot)[4]) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int32_t inc[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    inc[q] = v[q];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t t = __shfl_up_sync(0xffffffffu, inc[q], o);
      if (lane >= o) inc[q] += t;
    }
    if (lane == 31) sh[q][warp] = inc[q];
  }
  __syncthreads();
  if (warp == 0) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int32_t w = sh[q][lane];
      int32_t x = w;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int32_t t = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += t;
      }
      sh[q][lane] = x - w;              // exclusive prefix of the warp totals
      if (lane == 31) sh[q][32] = x;
    }
  }
  __syncthreads();
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    v[q] = sh[q][warp] + inc[q] - v[q];
    tot[q] = sh[q][32];
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kThreads, 1)
segments_kernel(const int32_t* __restrict__ token_adapter, int32_t T, const int32_t* __restrict__ rank,
                int32_t max_adapters, lora_segments seg, int32_t* __restrict__ err) {
  extern __shared__ int32_t sm[];
  int32_t* cnt = sm;                          // [K] tokens per key, then run starts / write cursors
  int32_t* krank = sm + (max_adapters + 1);   // [K] rank of the key's adapter
  __shared__ int32_t sh_scan[4][33];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int K = max_adapters + 1;              // key = adapter id + 1; key 0 = no adapter
  pdl_wait_then_release();

  for (int k = tid; k < K; k += kThreads) cnt[k] = 0;
  __syncthreads();

  // 1. validate ids, count tokens per key, remember each used adapter's rank
  for (int t = tid; t < T; t += kThreads) {
    const int32_t a = token_adapter[t];
    int32_t key = 0;
    if (a >= 0 && a < max_adapters) {
      const int32_t r = rank[a];
      if (r > 0) {
        key = a + 1;
        krank[key] = r;
      } else {
        flag_error(err, LORA_DEV_UNKNOWN_ADAPTER);
      }
    } else if (a != -1) {
      flag_error(err, LORA_DEV_UNKNOWN_ADAPTER);
    }
    seg.tok_adapter[t] = key - 1;
    atomicAdd(&cnt[key], 1);
  }
  __syncthreads();

  // 2. one scan gives run starts and segment indices, a second one the work-unit offsets
  //    inside each rank class; each thread then writes the segments and work units of its own
  //    keys.  Units are listed by rank class, largest ranks first (a unit's cost grows with
  //    the pages it gathers), then by adapter id and token offset, so that the delta kernel,
  //    which deals units to its clusters in waves, starts the longest ones first.
  const int per = (K + kThreads - 1) / kThreads;
  const int k_lo = min(K, tid * per), k_hi = min(K, k_lo + per);
  int32_t v[4] = {0, 0, 0, 0};                 // tokens, segments, -, -
  int32_t ub[4] = {0, 0, 0, 0};                // work units per rank class
  for (int k = k_lo; k < k_hi; ++k) {
    const int32_t c = cnt[k];
    v[0] += c;
    if (k > 0 && c > 0) {
      v[1] += 1;
      ub[rank_class(krank[k])] += (c + kUnitTokens - 1) / kUnitTokens;
    }
  }
  int32_t tot[4], utot[4];
  block_exclusive_scan4(v, sh_scan, tot);
  block_exclusive_scan4(ub, sh_scan, utot);
  ub[1] += utot[0];
  ub[2] += utot[0] + utot[1];
  ub[3] += utot[0] + utot[1] + utot[2];
  for (int k = k_lo; k < k_hi; ++k) {
    const int32_t c = cnt[k];
    if (k > 0 && c > 0) {
      const int32_t sidx = v[1];
      seg.seg_off[sidx] = v[0];
      seg.seg_adapter[sidx] = k - 1;
      const int32_t r = krank[k];
      int32_t& u = ub[rank_class(r)];
      for (int b = 0; b * kUnitTokens < c; ++b, ++u)
        reinterpret_cast<int4*>(seg.units)[u] =
            make_int4(k - 1, r, v[0] + b * kUnitTokens, min(kUnitTokens, c - b * kUnitTokens));
      ++v[1];
    }
    cnt[k] = v[0];                             // becomes the running write position of key k
    v[0] += c;
  }
  const int32_t S = tot[1];
  if (tid == 0) {
    seg.seg_off[S] = T;
    if (S == 0) seg.seg_off[0] = T;
    *seg.n_seg = S;
    *seg.n_units = utot[0] + utot[1] + utot[2] + utot[3];
  }
  __syncthreads();

  // 3. stable scatter, 1024 tokens at a time; the warps holding tokens take turns in index order
  for (int base_t = 0; base_t < T; base_t += kThreads) {
    const int t = base_t + tid;
    const bool valid = t < T;
    const int32_t key = valid ? seg.tok_adapter[t] + 1 : -1;
    const unsigned peers = __match_any_sync(0xffffffffu, key);
    const int lrank = __popc(peers & ((1u << lane) - 1u));
    const int leader = __ffs(peers) - 1;
    const int n_warps = min(kWarps, (T - base_t + 31) / 32);
    for (int w = 0; w < n_warps; ++w) {
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
}

}  // namespace

int launch_segments_build(const lora_pool* p, const int32_t* token_adapter, int32_t T, const lora_segments* seg,
                          cudaStream_t st, bool pdl) {
  const size_t smem = 2 * (size_t)(p->max_adapters + 1) * sizeof(int32_t);
  static DeviceFlags attr;
  int rc = ensure_smem_attr(attr, segments_kernel, (int)(2 * (LORA_MAX_ADAPTERS + 1) * sizeof(int32_t)),
                            "segments_kernel attribute");
  if (rc != LORA_OK) return rc;
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
