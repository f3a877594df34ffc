// Paged decode attention over the unified pool's KV pages.
//
// "S-LoRA, in depth", "Unified paging": a token's K and V at one layer are one H-vector page
// each, taken from the same free list as adapter pages (lora_kv_grow).  For one new token per
// request, at one layer, with heads of width D = H / n_heads:
//     s_j = q_h . K_{j,h} / sqrt(D),   p = softmax_j(s),   out_h = sum_j p_j V_{j,h}
// over the request's cached tokens j (plain scaled dot-product attention; the pages give no
// formula of their own).
//
// One CTA per (request, head), four warps splitting the cached tokens (token j to warp j % 4).
// Lane l holds dimensions [l * D/32, (l+1) * D/32) of the head: the head's slice of a K or V page
// is 2 D contiguous bytes, one coalesced load per warp.  The loop is bound by load latency: the
// CTA stages the page ids of kChunk tokens at a time in shared memory (one coalesced pass), and a
// warp issues the K and V slices of its next kBatch tokens before using any of them.  Each warp keeps a running maximum, the running sum of exp(s - max) and an fp32
// accumulator of V, rescaled when the maximum grows, taking its tokens in ascending order; the
// four warps' partial results merge in shared memory in warp order, and the output is rounded
// to bf16 once.  HBM-bound: 2 x tokens x 2 D bytes per (request, head).  Page ids are checked
// against the pool: a bad id sets the error word and its token is skipped.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <string>
#include <vector>

#include "lora_internal.h"

namespace {

constexpr int kWarps = 4;
constexpr int kBatch = 4;                          // tokens a warp has in flight
constexpr int kChunk = 512;                        // tokens whose page ids are staged at a time

__device__ __forceinline__ void flag_error(int32_t* err, int32_t bits) {
  atomicCAS(err, 0, LORA_EDEVICE);
  atomicOr(err + 1, bits);
}

// VPL consecutive bf16 values at p (8-byte aligned for VPL = 4, 4-byte for VPL = 2).
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

template <int D>
__global__ void __launch_bounds__(32 * kWarps)
attention_decode_kernel(const uint16_t* __restrict__ pool, int64_t num_pages, int32_t H,
                        const int32_t* __restrict__ table, int32_t max_len, int32_t layers, int32_t layer,
                        const int32_t* __restrict__ seq_len, const uint16_t* __restrict__ q,
                        uint16_t* __restrict__ out, int32_t n_heads, float scale, int32_t* err) {
  constexpr int VPL = D / 32;
  __shared__ float s_m[kWarps], s_l[kWarps];
  __shared__ float s_acc[kWarps][D];
  __shared__ int32_t s_ids[kChunk][2];               // (K page, V page) of the chunk's tokens
  const int req = blockIdx.y, h = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int n = seq_len[req];
  if (n < 0 || n > max_len) {
    if (threadIdx.x == 0) flag_error(err, LORA_DEV_BAD_SEGMENT);
    n = n < 0 ? 0 : max_len;
  }
  const int64_t col = (int64_t)h * D + lane * VPL;
  float qv[VPL];
  load_slice<VPL>(q + (int64_t)req * H + col, qv);
  float m = -INFINITY, l = 0.f, acc[VPL];
#pragma unroll
  for (int i = 0; i < VPL; ++i) acc[i] = 0.f;
  const int32_t* tab = table + (int64_t)req * max_len * layers * 2;
  for (int c0 = 0; c0 < n; c0 += kChunk) {
    const int cn = min(kChunk, n - c0);
    __syncthreads();                                 // the previous chunk's ids are consumed
    for (int i = threadIdx.x; i < 2 * cn; i += blockDim.x) {
      const int j = c0 + (i >> 1);
      s_ids[i >> 1][i & 1] = tab[((int64_t)j * layers + layer) * 2 + (i & 1)];
    }
    __syncthreads();
    for (int j0 = warp; j0 < cn; j0 += kWarps * kBatch) {
      // chunk tokens j0, j0 + 4, ..., j0 + 4 (kBatch - 1) of this warp: slices, then the math
      bool ok[kBatch];
      int32_t kp[kBatch], vp[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int j = j0 + u * kWarps;
        kp[u] = vp[u] = -1;
        if (j < cn) {
          kp[u] = s_ids[j][0];
          vp[u] = s_ids[j][1];
        }
      }
      float kv[kBatch][VPL], vv[kBatch][VPL];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int j = j0 + u * kWarps;
        ok[u] = kp[u] >= 0 && kp[u] < num_pages && vp[u] >= 0 && vp[u] < num_pages;   // same in every lane
        if (j < cn && !ok[u] && lane == 0) flag_error(err, LORA_DEV_BAD_PAGE);
        if (ok[u]) {
          load_slice<VPL>(pool + (int64_t)kp[u] * H + col, kv[u]);
          load_slice<VPL>(pool + (int64_t)vp[u] * H + col, vv[u]);
        }
      }
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        if (!ok[u]) continue;
        float s = 0.f;
#pragma unroll
        for (int i = 0; i < VPL; ++i) s = fmaf(qv[i], kv[u][i], s);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        s *= scale;
        const float m_new = fmaxf(m, s);
        const float c = expf(m - m_new);             // 0 on the first token (m = -inf)
        const float pj = expf(s - m_new);
        l = l * c + pj;
#pragma unroll
        for (int i = 0; i < VPL; ++i) acc[i] = fmaf(pj, vv[u][i], acc[i] * c);
        m = m_new;
      }
    }
  }
  if (lane == 0) {
    s_m[warp] = m;
    s_l[warp] = l;
  }
#pragma unroll
  for (int i = 0; i < VPL; ++i) s_acc[warp][lane * VPL + i] = acc[i];
  __syncthreads();
  if (warp == 0) {
    float M = -INFINITY;
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, s_m[w]);
    float L = 0.f, o[VPL];
#pragma unroll
    for (int i = 0; i < VPL; ++i) o[i] = 0.f;
    for (int w = 0; w < kWarps; ++w) {             // warps in order: a fixed summation order
      if (s_m[w] == -INFINITY) continue;           // the warp saw no token
      const float c = expf(s_m[w] - M);
      L = fmaf(s_l[w], c, L);
#pragma unroll
      for (int i = 0; i < VPL; ++i) o[i] = fmaf(s_acc[w][lane * VPL + i], c, o[i]);
    }
    uint16_t* dst = out + (int64_t)req * H + col;
#pragma unroll
    for (int i = 0; i < VPL; ++i)
      dst[i] = __bfloat16_as_ushort(__float2bfloat16_rn(L > 0.f ? o[i] / L : 0.f));
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
  const dim3 grid(n_heads, n_req);
  const float scale = 1.0f / std::sqrt((float)D);
  const uint16_t* pool = static_cast<const uint16_t*>(p->pool_dev);
  cudaError_t e;
  {
    ProfScope prof(p, LORA_KIND_ATTENTION, st);
    if (D == 128)
      attention_decode_kernel<128><<<grid, 32 * kWarps, 0, st>>>(pool, p->num_pages, p->H, table_dev, max_len, layers,
                                                                 layer, seq_len_dev, static_cast<const uint16_t*>(q),
                                                                 static_cast<uint16_t*>(out), n_heads, scale, p->d_err);
    else
      attention_decode_kernel<64><<<grid, 32 * kWarps, 0, st>>>(pool, p->num_pages, p->H, table_dev, max_len, layers,
                                                                layer, seq_len_dev, static_cast<const uint16_t*>(q),
                                                                static_cast<uint16_t*>(out), n_heads, scale, p->d_err);
    e = cudaGetLastError();
  }
  return e == cudaSuccess ? LORA_OK : lora_cuda_fail(e, "lora_attention_decode launch");
}
