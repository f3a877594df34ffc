// Segment builder: group a batch's tokens by adapter id, stably.
//
// The pages batch requests of many adapters into one base projection and gather each
// request's own A and B pages ("S-LoRA, in depth", section "The architecture"); grouping
// tokens by adapter lets each adapter's pages be read once per batch instead of once per
// token.  Output order: ascending adapter id, ties by token index; tokens without an
// adapter (-1) first and outside every segment.
//
// One CTA of 1024 threads: a shared-memory histogram over adapter ids (the rank table is
// read into shared memory beside it, while the first 1024 ids are in flight), one block scan
// that turns counts into run starts, segment indices and the offsets of the LoRA-delta work
// units within their rank class (each unit written right away as a complete record: adapter,
// rank, first index into perm, token count), then a stable scatter in chunks of 1024 tokens
// (warp-level match for ranks inside a warp, warps in order; the first chunk's keys stay in
// registers).
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

constexpr int kScanMax = 6;   // values per thread in one block scan, at most

// Exclusive block scan of N int32 values per thread; totals land in tot[0..N-1].
template <int N>
__device__ __forceinline__ void block_exclusive_scan(int32_t (&v)[N], int32_t (*sh)[33], int32_t (&tot)[N]) {
  static_assert(N <= kScanMax, "scan scratch holds kScanMax rows");
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int32_t inc[N];
#pragma unroll
  for (int q = 0; q < N; ++q) {
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
    for (int q = 0; q < N; ++q) {
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
  for (int q = 0; q < N; ++q) {
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
  __shared__ int32_t sh_scan[kScanMax][33];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int K = max_adapters + 1;              // key = adapter id + 1; key 0 = no adapter
  pdl_wait_then_release();

  const int32_t a_first = tid < T ? token_adapter[tid] : -1;   // in flight while the tables fill
  for (int k = tid; k < K; k += kThreads) {
    cnt[k] = 0;
    krank[k] = k > 0 ? rank[k - 1] : 0;
  }
  __syncthreads();

  // 1. validate ids, count tokens per key
  int32_t key_first = 0;                       // key of token tid, kept for the scatter
  for (int t = tid; t < T; t += kThreads) {
    const int32_t a = t == tid ? a_first : token_adapter[t];
    int32_t key = 0;
    if (a >= 0 && a < max_adapters) {
      if (krank[a + 1] > 0) key = a + 1;
      else flag_error(err, LORA_DEV_UNKNOWN_ADAPTER);
    } else if (a != -1) {
      flag_error(err, LORA_DEV_UNKNOWN_ADAPTER);
    }
    if (t == tid) key_first = key;
    seg.tok_adapter[t] = key - 1;
    atomicAdd(&cnt[key], 1);
  }
  __syncthreads();

  // 2. one scan gives run starts, segment indices and the work-unit offsets inside each rank
  //    class; each thread then writes the segments and work units of its own keys.  Units are
  //    listed by rank class, largest ranks first (a unit's cost grows with the pages it
  //    gathers), then by adapter id and token offset, so that the delta kernel, which deals
  //    units to its clusters in waves, starts the longest ones first.
  const int per = (K + kThreads - 1) / kThreads;
  const int k_lo = min(K, tid * per), k_hi = min(K, k_lo + per);
  int32_t v[6] = {0, 0, 0, 0, 0, 0};           // tokens, segments, work units per rank class
  for (int k = k_lo; k < k_hi; ++k) {
    const int32_t c = cnt[k];
    v[0] += c;
    if (k > 0 && c > 0) {
      v[1] += 1;
      v[2 + rank_class(krank[k])] += (c + kUnitTokens - 1) / kUnitTokens;
    }
  }
  int32_t tot[6];
  block_exclusive_scan(v, sh_scan, tot);
  const int32_t utot[4] = {tot[2], tot[3], tot[4], tot[5]};
  int32_t ub[4] = {v[2], v[3] + utot[0], v[4] + utot[0] + utot[1], v[5] + utot[0] + utot[1] + utot[2]};
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
    const int32_t key = !valid ? -1 : base_t == 0 ? key_first : seg.tok_adapter[t] + 1;
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
  if (seg.tile_plan == nullptr || T <= kTileTokens) return;

  // 4. tile plan of a prefill-shaped batch: the distinct adapters of every 256-token tile.  In
  //    perm (adapter-major, token order inside an adapter) the tokens of one adapter in one tile
  //    are a run; each run start names one (tile, adapter) pair.  Tiles with at most
  //    kTileAdapters adapters are fused, their adapters listed in ascending id order.
  __shared__ int32_t tile_cnt[LORA_MAX_TOKENS / kTileTokens];
  __shared__ int32_t tile_ad[LORA_MAX_TOKENS / kTileTokens][kTileAdapters];
  const int n_tiles = (T + kTileTokens - 1) / kTileTokens;
  for (int i = tid; i < n_tiles; i += kThreads) tile_cnt[i] = 0;
  __syncthreads();
  const int off0 = cnt[0];                     // the no-adapter tokens come first in perm
  for (int i = off0 + tid; i < T; i += kThreads) {
    const int32_t t = seg.perm[i];
    const int32_t a = seg.tok_adapter[t];
    bool first = i == off0;
    if (!first) {
      const int32_t tp = seg.perm[i - 1];
      first = seg.tok_adapter[tp] != a || (tp / kTileTokens) != (t / kTileTokens);
    }
    if (first) {
      const int tile = t / kTileTokens;
      const int b = atomicAdd(&tile_cnt[tile], 1);
      if (b < kTileAdapters) tile_ad[tile][b] = a;
    }
  }
  __syncthreads();
  int32_t ev[4] = {0, 0, 0, 0};                // fused (tile, adapter) pairs of this thread's tile
  int32_t nb = 0;
  if (tid < n_tiles) {
    nb = tile_cnt[tid] <= kTileAdapters ? tile_cnt[tid] : -1;
    int32_t ad[kTileAdapters];
#pragma unroll
    for (int b = 0; b < kTileAdapters; ++b) ad[b] = b < nb ? tile_ad[tid][b] : -1;
#pragma unroll
    for (int i = 1; i < kTileAdapters; ++i)    // insertion sort of at most 4 ids
#pragma unroll
      for (int j = i; j > 0; --j)
        if (j < nb && ad[j - 1] > ad[j]) {
          const int32_t x = ad[j - 1];
          ad[j - 1] = ad[j];
          ad[j] = x;
        }
    int32_t* pl = seg.tile_plan + (size_t)tid * kPlanStride;
    pl[0] = nb;
#pragma unroll
    for (int b = 0; b < kTileAdapters; ++b) pl[1 + b] = ad[b];
    ev[0] = nb > 0 ? nb : 0;
  }
  for (int i = n_tiles + tid; i < seg.n_tiles_max; i += kThreads) seg.tile_plan[(size_t)i * kPlanStride] = -1;
  int32_t etot[4];
  block_exclusive_scan(ev, sh_scan, etot);    // also orders the tile_cnt reads before the rewrite below
  if (tid < n_tiles) {
    for (int b = 0; b < nb; ++b) seg.entries[ev[0] + b] = tid * kTileAdapters + b;
    tile_cnt[tid] = nb;                        // from here on: < 0 marks a tile that is not fused
  }
  if (tid == 0) *seg.n_entries = etot[0];
  __syncthreads();

  // 5. the work units the LoRA-delta kernel still has to do when the fused tiles take their
  //    LoRA term in the GEMM: those holding a token of a tile that is not fused, kept in order;
  //    a unit that also holds tokens of fused tiles gets kUnitMixed in its token count, so the
  //    delta kernel looks tiles up only for such units.
  const int32_t n_units = utot[0] + utot[1] + utot[2] + utot[3];
  const int u_per = (n_units + kThreads - 1) / kThreads;
  const int u_lo = min(n_units, tid * u_per), u_hi = min(n_units, u_lo + u_per);
  int32_t lv[4] = {0, 0, 0, 0};
  uint32_t live_bits = 0, mixed_bits = 0;      // u_per <= 32 for every T <= LORA_MAX_TOKENS
  for (int u = u_lo; u < u_hi; ++u) {
    const int4 rec = reinterpret_cast<const int4*>(seg.units)[u];
    bool live = false, fused = false;
    for (int j = 0; j < rec.w; ++j) {
      const bool f = tile_cnt[seg.perm[rec.z + j] / kTileTokens] >= 0;
      live = live || !f;
      fused = fused || f;
    }
    if (live) {
      live_bits |= 1u << (u - u_lo);
      if (fused) mixed_bits |= 1u << (u - u_lo);
      ++lv[0];
    }
  }
  int32_t ltot[4];
  block_exclusive_scan(lv, sh_scan, ltot);
  for (int u = u_lo, pos = lv[0]; u < u_hi; ++u)
    if ((live_bits >> (u - u_lo)) & 1u) {
      int4 rec = reinterpret_cast<const int4*>(seg.units)[u];
      if ((mixed_bits >> (u - u_lo)) & 1u) rec.w |= kUnitMixed;
      reinterpret_cast<int4*>(seg.units_rest)[pos++] = rec;
    }
  if (tid == 0) *seg.n_units_rest = ltot[0];
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
