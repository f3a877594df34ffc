// lora_linear_forward: one projection slot of the unmerged multi-adapter layer.
// lora_linear_forward_group: several slots that read the same input (q, k and v of a layer).
//
// "S-LoRA, in depth", section "Merge or keep adapters separate": y = xW + (xA)B per token,
// W shared, A and B the token's own adapter.  Kernels on the caller's stream:
//   1. LoRA delta: s = x A, then delta = s B, per run of tokens sharing an adapter (paged
//      gathers, fused in one kernel; s stays on chip), for every slot of the call at once
//   2. base GEMM x W^T on tcgen05, epilogue y = bf16_rne(acc + delta): one launch per slot, or
//      for a group of slots and a batch of <= 256 tokens one persistent launch over all of them
#include <cuda_runtime.h>

#include <string>

#include "lora_internal.h"

namespace {

int forward_slots(lora_pool* p, const lora_segments* seg, int32_t n, const int32_t* slots, const void* x,
                  const void* const* W, void* const* y, float* const* delta_dbg, lora_stream_t stream,
                  const char* name) {
  const std::string fn(name);
  if (!p || !seg) return lora_fail(LORA_EINVAL, fn + ": pool or segments is NULL");
  if (p->planning) return lora_fail(LORA_EINVAL, fn + ": planning pool has no device state");
  const int32_t cap = seg->delta_slots > 1 ? seg->delta_slots : 1;
  if (n < 1 || n > LORA_MAX_GROUP || n > cap)
    return lora_fail(LORA_EINVAL, fn + ": " + std::to_string(n) + " slots, the workspace holds delta scratch for " +
                                      std::to_string(cap));
  if (!slots || !W || !y) return lora_fail(LORA_EINVAL, fn + ": slot, W and y arrays are required");
  for (int i = 0; i < n; ++i) {
    if (slots[i] < 0 || slots[i] >= p->n_slots) return lora_fail(LORA_EINVAL, fn + ": slot out of range");
    for (int j = 0; j < i; ++j)
      if (slots[j] == slots[i]) return lora_fail(LORA_EINVAL, fn + ": a slot is listed twice");
  }
  if (seg->T < 0) return lora_fail(LORA_EINVAL, fn + ": no batch built into the segments");
  if (seg->H != p->H) return lora_fail(LORA_EINVAL, fn + ": segments sized for another pool");
  const int32_t T = seg->T, H = p->H;
  if (T == 0) return LORA_OK;
  if (!x) return lora_fail(LORA_EINVAL, fn + ": x, W and y are required");
  for (int i = 0; i < n; ++i) {
    if (!W[i] || !y[i]) return lora_fail(LORA_EINVAL, fn + ": x, W and y are required");
    const uintptr_t mis = reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(W[i]) |
                          reinterpret_cast<uintptr_t>(y[i]) |
                          reinterpret_cast<uintptr_t>(delta_dbg ? delta_dbg[i] : nullptr);
    if (mis & 15) return lora_fail(LORA_EINVAL, fn + ": x, W, y and delta must be 16-byte aligned");
    if (x == y[i]) return lora_fail(LORA_EINVAL, fn + ": y must not alias x");
    for (int j = 0; j < i; ++j)
      if (y[j] == y[i]) return lora_fail(LORA_EINVAL, fn + ": two slots share one y");
  }
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);

  LoraLaunch L = {};
  L.pool = static_cast<const uint16_t*>(p->pool_dev);
  L.num_pages = p->num_pages;
  L.H = H;
  L.T = T;
  L.n_slots = p->n_slots;
  L.n_group = n;
  for (int i = 0; i < n; ++i) {
    float* dbg = delta_dbg ? delta_dbg[i] : nullptr;
    L.slot[i] = slots[i];
    L.delta[i] = dbg ? dbg : seg->delta + (size_t)i * seg->T_max * H;
    if (dbg) {
      cudaError_t e = cudaMemsetAsync(dbg, 0, (size_t)T * H * sizeof(float), st);
      if (e != cudaSuccess) return lora_cuda_fail(e, "lora_linear_forward: clearing delta");
    }
  }
  L.ptab = p->d_ptab;
  L.rank = p->d_rank;
  L.seg = seg;
  L.x = static_cast<const uint16_t*>(x);
  L.err = p->d_err;
  L.pdl = !p->prof_on;
  int rc;
  {
    ProfScope prof(p, LORA_KIND_DELTA, st);
    rc = launch_lora_delta(L, st);
  }
  if (rc != LORA_OK) return rc;

  GemmLaunch G[LORA_MAX_GROUP];
  for (int i = 0; i < n; ++i) {
    G[i].x = static_cast<const uint16_t*>(x);
    G[i].W = static_cast<const uint16_t*>(W[i]);
    G[i].y = static_cast<uint16_t*>(y[i]);
    G[i].delta = L.delta[i];
    G[i].tok_adapter = seg->tok_adapter;
    G[i].ptab = p->d_ptab;
    G[i].T = T;
    G[i].H = H;
    G[i].slot = slots[i];
    G[i].n_slots = p->n_slots;
    G[i].partials = seg->gemm_partials;
    G[i].partials_floats = gemm_partial_floats(seg->T_max, H) * cap;
    G[i].err = p->d_err;
    G[i].pdl = !p->prof_on;
  }
  if (gemm_group_fits(G, n)) {          // decode-sized batch: one launch for every slot of the group
    ProfScope prof(p, LORA_KIND_GEMM, st);
    return launch_gemm_group(G, n, st);
  }
  for (int i = 0; i < n; ++i) {
    ProfScope prof(p, LORA_KIND_GEMM, st);
    rc = launch_gemm(G[i], st);
    if (rc != LORA_OK) return rc;
  }
  return LORA_OK;
}

}  // namespace

extern "C" int lora_linear_forward(lora_pool* p, const lora_segments* seg, int32_t slot, const void* x, const void* W,
                                   void* y, float* delta_dbg, lora_stream_t stream) {
  return forward_slots(p, seg, 1, &slot, x, &W, &y, &delta_dbg, stream, "lora_linear_forward");
}

extern "C" int lora_linear_forward_group(lora_pool* p, const lora_segments* seg, int32_t n, const int32_t* slots_host,
                                         const void* x, const void* const* W_host, void* const* y_host,
                                         float* const* delta_dbg_host, lora_stream_t stream) {
  return forward_slots(p, seg, n, slots_host, x, W_host, y_host, delta_dbg_host, stream, "lora_linear_forward_group");
}
