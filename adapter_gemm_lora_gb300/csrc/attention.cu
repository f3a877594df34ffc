// Paged decode attention over the unified pool's KV pages.
//
// "S-LoRA, in depth", "Unified paging": a token's K and V at one layer are one H-vector page
// each, taken from the same free list as adapter pages (lora_kv_grow).  For one new token per
// request, at one layer, with heads of width D = H / n_heads:
//     s_j = q_h . K_{j,h} / sqrt(D),   p = softmax_j(s),   out_h = sum_j p_j V_{j,h}
// over the request's cached tokens j (plain scaled dot-product attention; the pages give no
// formula of their own).
//
// One CTA per (group of 8 heads, request) reads, per cached token, the group's slice of the K
// page row and of the V page row (8 D contiguous bf16 each) with cp.async.bulk into a ring of
// shared-memory stages of 8 tokens, one mbarrier transaction count per stage; a warp per head
// keeps its running maximum, running sum of exp and fp32 accumulator of V in registers and takes
// the tokens in ascending order, 8 at a time (the running values are updated once per batch).
// The output is rounded to bf16 once.  HBM-bound: 2 x tokens x 2 H bytes per request.  Page ids
// are checked against the pool: a bad id sets the error word and its token is skipped.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <string>
#include <vector>

#include "tc_ptx.h"

namespace {

// VPL consecutive bf16 values at p, global or shared (8-byte aligned for VPL = 4, 4-byte for VPL = 2).
template <int VPL>
__device__ __forceinline__ void load_slice(const uint16_t* p, float (&v)[VPL]) {
  if constexpr (VPL == 4) {
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    v[0] = __uint_as_float(u.x << 16);
    v[1] = __uint_as_float(u.x & 0xFFFF0000u);
    v[2] = __uint_as_float(u.y << 16);
    v[3] = __uint_as_float(u.y & 0xFFFF0000u);
  } else {
    const uint32_t u = *reinterpret_cast<const uint32_t*>(p);
    v[0] = __uint_as_float(u << 16);
    v[1] = __uint_as_float(u & 0xFFFF0000u);
  }
}

// ---- head-group kernel -----------------------------------------------------------------------
constexpr int kGroupHeads = 8;                        // heads a CTA takes, one per consumer warp
constexpr int kTokBatch = 8;                          // tokens in a ring stage
constexpr int kGrpStages = 3;                         // ring stages
constexpr int kGrpThreads = 32 * (kGroupHeads + 1);   // + the producer warp

// Shared memory: kGrpStages stages of kTokBatch tokens' [K slice | V slice] (8 D bf16 each), the
// full and empty mbarriers (8-byte aligned: the ring is a multiple of 1 KB), then the mask of
// tokens with data per stage.  96 KB of ring at D = 128.
template <int D>
constexpr size_t grp_smem_bytes() {
  return (size_t)kGrpStages * kTokBatch * (2 * kGroupHeads * D * 2) + 2 * kGrpStages * 8 + kGrpStages * 4;
}

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

// Sums eight per-lane values over the warp with 9 shuffles: on return, lane l holds the sum of
// value t(l) = 4 b4 + 2 b3 + b2 (b_i: bit i of l).  Each step halves the values a lane keeps,
// trading the other half with its partner (xor 16, 8, 4), and the last two steps add within
// groups of four lanes; partners add the same two numbers, so all lanes of a group agree bitwise.
__device__ __forceinline__ float reduce8_transpose(const float (&v)[kTokBatch], int lane) {
  float w[4], u[2];
  const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float keep = b4 ? v[i + 4] : v[i], send = b4 ? v[i] : v[i + 4];
    w[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float keep = b3 ? w[i + 2] : w[i], send = b3 ? w[i] : w[i + 2];
    u[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
  }
  float z = (b2 ? u[1] : u[0]) + __shfl_xor_sync(0xffffffffu, b2 ? u[0] : u[1], 4);
  z += __shfl_xor_sync(0xffffffffu, z, 2);
  z += __shfl_xor_sync(0xffffffffu, z, 1);
  return z;
}

// One CTA per (group of 8 heads, request).  Warp 8 fills the ring a batch of 8 tokens at a time:
// lane u < 8 copies token u's slice of its K page row and of its V page row (8 D bf16 each, 2 KB
// at D = 128) with cp.async.bulk, all against the stage's one mbarrier.  Warp w < 8 owns head
// 8 g + w: per batch, eight partial dot products per lane, one transposing reduction, each lane's
// exp2 for its token, then the V rows with the eight weights.  Softmax in base 2: scores carry
// log2(e) / sqrt(D), and the running maximum and sum are updated once per batch.
template <int D>
__global__ void __launch_bounds__(kGrpThreads)
attention_heads_kernel(const uint16_t* __restrict__ pool, int64_t num_pages, int32_t H,
                       const int32_t* __restrict__ table, int32_t max_len, int32_t layers, int32_t layer,
                       const int32_t* __restrict__ seq_len, const uint16_t* __restrict__ q,
                       uint16_t* __restrict__ out, int32_t n_heads, float scale_log2, int32_t* err) {
  constexpr int VPL = D / 32;
  constexpr uint32_t kRow = kGroupHeads * D * 2;      // bytes of a K (or V) slice slot
  constexpr uint32_t kTok = 2 * kRow;                 // one token: K slot then V slot
  constexpr uint32_t kStage = kTokBatch * kTok;
  extern __shared__ __align__(128) uint8_t smem[];
  static_assert(kStage % 1024 == 0, "the mbarriers after the ring must be 8-byte aligned");
  const uint32_t bar_full = smem_u32(smem + (size_t)kGrpStages * kStage);
  const uint32_t bar_empty = bar_full + 8 * kGrpStages;
  uint32_t* vmask_s = reinterpret_cast<uint32_t*>(smem + (size_t)kGrpStages * kStage + 2 * kGrpStages * 8);
  const uint32_t ring = smem_u32(smem);
  const int req = blockIdx.y, h0 = blockIdx.x * kGroupHeads;
  const int n_act = min(kGroupHeads, n_heads - h0);   // heads of this group
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int n = seq_len[req];
  if (n < 0 || n > max_len) {
    if (threadIdx.x == 0) flag_error(err, LORA_DEV_BAD_SEGMENT);
    n = n < 0 ? 0 : max_len;
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < kGrpStages; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, n_act);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  const int n_batches = (n + kTokBatch - 1) / kTokBatch;

  if (warp == kGroupHeads) {
    // ---- producer: batch b into stage b % kGrpStages ----
    const int32_t* tab = table + (int64_t)req * max_len * layers * 2;
    const uint32_t bytes = (uint32_t)n_act * D * 2;
    bool ok = true;
    int b = 0;
    for (; b < n_batches; ++b) {
      const int s = b % kGrpStages, j = b * kTokBatch + lane;
      int32_t kp = -1, vp = -1;
      if (lane < kTokBatch && j < n) {
        kp = tab[((int64_t)j * layers + layer) * 2];
        vp = tab[((int64_t)j * layers + layer) * 2 + 1];
      }
      const bool valid = kp >= 0 && kp < num_pages && vp >= 0 && vp < num_pages;
      const uint32_t vm = __ballot_sync(0xffffffffu, valid);
      if (lane < kTokBatch && j < n && !valid) flag_error(err, LORA_DEV_BAD_PAGE);   // the token is skipped
      ok = __all_sync(0xffffffffu, mbar_wait(bar_empty + 8 * s, ((b / kGrpStages) & 1) ^ 1));
      if (!ok) break;
      if (lane == 0) {
        vmask_s[s] = vm;
        mbar_arrive_expect_tx(bar_full + 8 * s, 2 * bytes * __popc(vm));
      }
      __syncwarp();
      if (valid) {
        const uint32_t dst = ring + (uint32_t)s * kStage + (uint32_t)lane * kTok;
        bulk_g2s(dst, pool + (int64_t)kp * H + h0 * D, bytes, bar_full + 8 * s);
        bulk_g2s(dst + kRow, pool + (int64_t)vp * H + h0 * D, bytes, bar_full + 8 * s);
      }
    }
    if (!ok && lane == 0) {
      flag_error(err, LORA_DEV_WAIT_TIMEOUT);
      // the copies already issued land before this CTA's shared memory is released
      for (int c = b > kGrpStages ? b - kGrpStages : 0; c < b; ++c)
        (void)mbar_wait(bar_full + 8 * (c % kGrpStages), (c / kGrpStages) & 1);
    }
  } else if (warp < n_act) {
    // ---- consumer: head h0 + warp ----
    const int hd = warp * D + lane * VPL;              // this lane's offset in a slice
    float qv[VPL], acc[VPL];
    load_slice<VPL>(q + (int64_t)req * H + (int64_t)h0 * D + hd, qv);
#pragma unroll
    for (int k = 0; k < VPL; ++k) acc[k] = 0.f;
    float m = -INFINITY, l = 0.f;
    const int t_lane = ((lane >> 4) & 1) * 4 + ((lane >> 3) & 1) * 2 + ((lane >> 2) & 1);
    bool ok = true;
    for (int b = 0; b < n_batches; ++b) {
      const int s = b % kGrpStages;
      ok = __all_sync(0xffffffffu, mbar_wait(bar_full + 8 * s, (b / kGrpStages) & 1));
      if (!ok) break;
      const uint32_t vmask = vmask_s[s];               // tokens of the batch with data
      const uint8_t* st = smem + (size_t)s * kStage;
      float part[kTokBatch];
#pragma unroll
      for (int g = 0; g < kTokBatch; ++g) {
        part[g] = 0.f;
        if ((vmask >> g) & 1u) {
          float kv[VPL];
          load_slice<VPL>(reinterpret_cast<const uint16_t*>(st + g * kTok) + hd, kv);
#pragma unroll
          for (int k = 0; k < VPL; ++k) part[g] = fmaf(qv[k], kv[k], part[g]);
        }
      }
      const float z = reduce8_transpose(part, lane);
      const float sc = ((vmask >> t_lane) & 1u) ? z * scale_log2 : -INFINITY;
      float mb = fmaxf(sc, __shfl_xor_sync(0xffffffffu, sc, 4));
      mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 8));
      mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 16));
      const float m_new = fmaxf(m, mb);
      if (m_new != -INFINITY) {                        // same in every lane
        const float c = exp2f(m - m_new);              // 0 while no token has been seen
        const float p = exp2f(sc - m_new);             // this lane's token; 0 for a token without data
        float ps = p + __shfl_xor_sync(0xffffffffu, p, 4);
        ps += __shfl_xor_sync(0xffffffffu, ps, 8);
        ps += __shfl_xor_sync(0xffffffffu, ps, 16);
        l = fmaf(l, c, ps);
#pragma unroll
        for (int k = 0; k < VPL; ++k) acc[k] *= c;
#pragma unroll
        for (int g = 0; g < kTokBatch; ++g) {
          const float pg = __shfl_sync(0xffffffffu, p, ((g >> 2) << 4) | (((g >> 1) & 1) << 3) | ((g & 1) << 2));
          if ((vmask >> g) & 1u) {
            float vv[VPL];
            load_slice<VPL>(reinterpret_cast<const uint16_t*>(st + g * kTok + kRow) + hd, vv);
#pragma unroll
            for (int k = 0; k < VPL; ++k) acc[k] = fmaf(pg, vv[k], acc[k]);
          }
        }
        m = m_new;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_empty + 8 * s);
    }
    if (!ok && lane == 0) flag_error(err, LORA_DEV_WAIT_TIMEOUT);
    uint16_t* dst = out + (int64_t)req * H + (int64_t)h0 * D + hd;
#pragma unroll
    for (int k = 0; k < VPL; ++k)
      dst[k] = __bfloat16_as_ushort(__float2bfloat16_rn(l > 0.f ? acc[k] / l : 0.f));
  }
}

}  // namespace

extern "C" int lora_kv_batch_table(lora_pool* p, const int64_t* request_ids, int32_t n_req, int32_t max_len,
                                   int32_t* table_dev, int32_t* seq_len_dev, lora_stream_t stream) {
  if (!p || n_req < 0 || max_len < 0 || (n_req > 0 && (!request_ids || !table_dev || !seq_len_dev)))
    return lora_fail(LORA_EINVAL, "lora_kv_batch_table: bad arguments");
  if (p->planning) return lora_fail(LORA_EINVAL, "lora_kv_batch_table: planning pool has no device state");
  if (n_req == 0) return LORA_OK;
  int32_t layers = -1;
  for (int i = 0; i < n_req; ++i) {
    auto it = p->kv.find(request_ids[i]);
    if (it == p->kv.end())
      return lora_fail(LORA_EINVAL, "lora_kv_batch_table: request " + std::to_string(request_ids[i]) + " holds no pages");
    if (layers < 0) layers = it->second.layers;
    if (it->second.layers != layers)
      return lora_fail(LORA_EINVAL, "lora_kv_batch_table: requests with different layer counts");
    if ((int64_t)it->second.pages.size() / (2 * layers) > max_len)
      return lora_fail(LORA_EINVAL, "lora_kv_batch_table: a request holds more than max_len tokens");
  }
  const size_t per_req = (size_t)max_len * layers * 2;
  p->h_kvtab.assign(per_req * n_req + n_req, -1);
  int32_t* lens = p->h_kvtab.data() + per_req * n_req;
  for (int i = 0; i < n_req; ++i) {
    const auto& pages = p->kv.find(request_ids[i])->second.pages;
    std::copy(pages.begin(), pages.end(), p->h_kvtab.begin() + per_req * i);
    lens[i] = (int32_t)(pages.size() / (2 * layers));
  }
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(table_dev, p->h_kvtab.data(), per_req * n_req * sizeof(int32_t),
                                  cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(seq_len_dev, lens, n_req * sizeof(int32_t), cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);      // the host table is reused by the next call
  return e == cudaSuccess ? LORA_OK : lora_cuda_fail(e, "lora_kv_batch_table");
}

extern "C" int lora_attention_decode(lora_pool* p, int32_t n_req, const int32_t* table_dev, const int32_t* seq_len_dev,
                                     int32_t max_len, int32_t layers, int32_t layer, const void* q, void* out,
                                     int32_t n_heads, lora_stream_t stream) {
  if (!p || n_req < 0 || max_len < 0 || layers < 1 || layer < 0 || layer >= layers || n_heads < 1)
    return lora_fail(LORA_EINVAL, "lora_attention_decode: bad arguments");
  if (p->planning) return lora_fail(LORA_EINVAL, "lora_attention_decode: planning pool has no device state");
  if (n_req == 0) return LORA_OK;
  if (!table_dev || !seq_len_dev || !q || !out) return lora_fail(LORA_EINVAL, "lora_attention_decode: null pointer");
  if (p->H % n_heads != 0) return lora_fail(LORA_EINVAL, "lora_attention_decode: H is not a multiple of n_heads");
  const int D = p->H / n_heads;
  if (D != 64 && D != 128) return lora_fail(LORA_EINVAL, "lora_attention_decode: head width must be 64 or 128");
  if (((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(out)) & 15) != 0)
    return lora_fail(LORA_EINVAL, "lora_attention_decode: q and out must be 16-byte aligned");
  if (n_req > 65535) return lora_fail(LORA_EINVAL, "lora_attention_decode: at most 65535 requests per call");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const uint16_t* pool = static_cast<const uint16_t*>(p->pool_dev);
  const float scale_log2 = 1.4426950408889634f / std::sqrt((float)D);   // log2(e) / sqrt(D)
  const dim3 grid((n_heads + kGroupHeads - 1) / kGroupHeads, n_req);
  const auto run = [&](auto kernel, size_t smem) -> cudaError_t {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    ProfScope prof(p, LORA_KIND_ATTENTION, st);
    kernel<<<grid, kGrpThreads, smem, st>>>(pool, p->num_pages, p->H, table_dev, max_len, layers, layer, seq_len_dev,
                                            static_cast<const uint16_t*>(q), static_cast<uint16_t*>(out), n_heads,
                                            scale_log2, p->d_err);
    return cudaGetLastError();
  };
  const cudaError_t e = D == 128 ? run(attention_heads_kernel<128>, grp_smem_bytes<128>())
                                 : run(attention_heads_kernel<64>, grp_smem_bytes<64>());
  return e == cudaSuccess ? LORA_OK : lora_cuda_fail(e, "lora_attention_decode launch");
}
