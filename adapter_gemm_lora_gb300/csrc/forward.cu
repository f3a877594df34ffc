// lora_linear_forward: one projection slot of the unmerged multi-adapter layer.
//
// "S-LoRA, in depth", section "Merge or keep adapters separate": y = xW + (xA)B per token,
// W shared, A and B the token's own adapter.  Three kernels on the caller's stream:
//   1. LoRA delta: s = x A, then delta = s B, per run of tokens sharing an adapter (paged
//      gathers, fused in one kernel; s stays on chip)
//   2. base GEMM x W^T on tcgen05, epilogue y = bf16_rne(acc + delta)
#include <cuda_runtime.h>

#include "lora_internal.h"

extern "C" int lora_linear_forward(lora_pool* p, const lora_segments* seg, int32_t slot, const void* x, const void* W,
                                   void* y, float* delta_dbg, lora_stream_t stream) {
  if (!p || !seg) return lora_fail(LORA_EINVAL, "lora_linear_forward: pool or segments is NULL");
  if (p->planning) return lora_fail(LORA_EINVAL, "lora_linear_forward: planning pool has no device state");
  if (slot < 0 || slot >= p->n_slots) return lora_fail(LORA_EINVAL, "lora_linear_forward: slot out of range");
  if (seg->T < 0) return lora_fail(LORA_EINVAL, "lora_linear_forward: no batch built into the segments");
  if (seg->H != p->H) return lora_fail(LORA_EINVAL, "lora_linear_forward: segments sized for another pool");
  const int32_t T = seg->T, H = p->H;
  if (T == 0) return LORA_OK;
  if (!x || !W || !y) return lora_fail(LORA_EINVAL, "lora_linear_forward: x, W and y are required");
  const uintptr_t mis = reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(W) | reinterpret_cast<uintptr_t>(y) |
                        reinterpret_cast<uintptr_t>(delta_dbg);
  if (mis & 15) return lora_fail(LORA_EINVAL, "lora_linear_forward: x, W, y and delta must be 16-byte aligned");
  if (x == y) return lora_fail(LORA_EINVAL, "lora_linear_forward: y must not alias x");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);

  float* delta = delta_dbg ? delta_dbg : seg->delta;
  if (delta_dbg) {
    cudaError_t e = cudaMemsetAsync(delta_dbg, 0, (size_t)T * H * sizeof(float), st);
    if (e != cudaSuccess) return lora_cuda_fail(e, "lora_linear_forward: clearing delta");
  }
  LoraLaunch L;
  L.pool = static_cast<const uint16_t*>(p->pool_dev);
  L.num_pages = p->num_pages;
  L.H = H;
  L.T = T;
  L.slot = slot;
  L.n_slots = p->n_slots;
  L.ptab = p->d_ptab;
  L.rank = p->d_rank;
  L.seg = seg;
  L.x = static_cast<const uint16_t*>(x);
  L.delta = delta;
  L.err = p->d_err;
  L.pdl = !p->prof_on;
  int rc;
  {
    ProfScope prof(p, LORA_KIND_DELTA, st);
    rc = launch_lora_delta(L, st);
  }
  if (rc != LORA_OK) return rc;

  GemmLaunch G;
  G.x = static_cast<const uint16_t*>(x);
  G.W = static_cast<const uint16_t*>(W);
  G.y = static_cast<uint16_t*>(y);
  G.delta = delta;
  G.tok_adapter = seg->tok_adapter;
  G.ptab = p->d_ptab;
  G.T = T;
  G.H = H;
  G.slot = slot;
  G.n_slots = p->n_slots;
  G.partials = seg->gemm_partials;
  G.partials_floats = gemm_partial_floats(seg->T_max, H);
  G.err = p->d_err;
  G.pdl = !p->prof_on;
  ProfScope prof(p, LORA_KIND_GEMM, st);
  return launch_gemm(G, st);
}
