// lora_linear_forward: one projection slot of the unmerged multi-adapter layer.
// lora_linear_forward_group: several slots that read the same input (q, k and v of a layer).
//
// "S-LoRA, in depth", section "Merge or keep adapters separate": y = xW + (xA)B per token,
// W shared, A and B the token's own adapter.  Kernels on the caller's stream:
//   1. LoRA delta: s = x A, then delta = s B, per run of tokens sharing an adapter (paged
//      gathers, fused in one kernel; s stays on chip), for every slot of the call at once
//   2. base GEMM x W^T on tcgen05, epilogue y = bf16_rne(acc + delta): one launch per slot, or
//      one launch for a group of slots
// A prefill-shaped batch (more than 256 tokens, on the persistent GEMM) is cut into 256-token
// tiles; the tiles with at most LORA_TILE_ADAPTERS adapters ("fused", planned by the segment
// build) take their LoRA term inside the GEMM instead ("Kernels for a batch of mixed ranks": many
// tokens share each adapter there, so the expand is a dense product per tile):
//   1. LoRA delta for the tokens of the other tiles only
//   2. shrink of the fused tiles on tcgen05: s = x A as bf16 hi + lo parts
//   3. (delta_dbg only) the GEMM's LoRA extension alone, fp32 into delta_dbg for the fused tiles
//   4. base GEMM whose accumulator of a fused tile also takes s B (B pages read through the
//      page table), y = bf16_rne(acc) there; other tiles add the delta as above
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

  GemmLaunch G[LORA_MAX_GROUP];
  for (int i = 0; i < n; ++i) {
    G[i] = GemmLaunch{};
    G[i].x = static_cast<const uint16_t*>(x);
    G[i].W = static_cast<const uint16_t*>(W[i]);
    G[i].y = static_cast<uint16_t*>(y[i]);
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
    G[i].prof = p;
    if (seg->tile_plan != nullptr && T > kTileTokens) {
      G[i].tile_plan = seg->tile_plan;
      G[i].s_lora = seg->s_lora + (size_t)i * seg->T_max * kSCols;
      G[i].pool = static_cast<const uint16_t*>(p->pool_dev);
      G[i].num_pages = p->num_pages;
      G[i].rank = p->d_rank;
    }
  }
  const bool fused = gemm_fused_fits(G, n);

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
  L.units = fused ? seg->units_rest : seg->units;
  L.n_units = fused ? seg->n_units_rest : seg->n_units;
  L.tile_plan = fused ? seg->tile_plan : nullptr;
  L.x = static_cast<const uint16_t*>(x);
  L.err = p->d_err;
  L.pdl = !p->prof_on;
  int rc;
  {
    ProfScope prof(p, LORA_KIND_DELTA, st);
    rc = launch_lora_delta(L, st);
  }
  if (rc != LORA_OK) return rc;
  for (int i = 0; i < n; ++i) G[i].delta = L.delta[i];

  if (fused) {
    ShrinkLaunch S = {};
    S.pool = L.pool;
    S.num_pages = p->num_pages;
    S.H = H;
    S.T = T;
    S.n_slots = p->n_slots;
    S.n_group = n;
    for (int i = 0; i < n; ++i) S.slot[i] = slots[i];
    S.ptab = p->d_ptab;
    S.rank = p->d_rank;
    S.seg = seg;
    S.x = L.x;
    S.err = p->d_err;
    S.pdl = L.pdl;
    {
      ProfScope prof(p, LORA_KIND_SHRINK, st);
      rc = launch_lora_shrink(S, st);
    }
    if (rc != LORA_OK) return rc;
    if (delta_dbg != nullptr) {         // the fused tiles' LoRA term, as the GEMM computes it, alone
      bool any = false;
      for (int i = 0; i < n; ++i) {
        G[i].lora_dbg = delta_dbg[i] ? delta_dbg[i] : seg->delta + (size_t)i * seg->T_max * H;
        any = any || delta_dbg[i] != nullptr;
      }
      if (any) {
        rc = launch_gemm_fused(G, n, true, st);
        if (rc != LORA_OK) return rc;
      }
    }
    return launch_gemm_fused(G, n, false, st);       // each GEMM kernel launch is its own profiling scope
  }
  if (gemm_group_fits(G, n)) return launch_gemm_group(G, n, st);   // decode-sized batch: one launch for the group
  for (int i = 0; i < n; ++i) {
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
