// Expert routing shared by the router kernels and the expert gate/up kernel:
// softmax + top-k of one row and the per-expert pair permutation. Both are
// pure functions of the router logits, so every kernel that runs them gets the
// same routing bits.
#pragma once
#include "common.cuh"

namespace spec {

// Softmax over E <= 256 logits and the top-k of one row, by one warp.
__device__ __forceinline__ void router_topk(const float* logit, int E, int k, int* ids, float* wts) {
  const int lane = threadIdx.x & 31;
  constexpr int MAXE = 8;
  float v[MAXE];
  float m = -INFINITY;
#pragma unroll
  for (int i = 0; i < MAXE; ++i) {
    const int e = lane + 32 * i;
    v[i] = e < E ? logit[e] : -INFINITY;
    m = fmaxf(m, v[i]);
  }
  m = warp_max(m);
  float z = 0.f;
#pragma unroll
  for (int i = 0; i < MAXE; ++i) {
    v[i] = (lane + 32 * i < E) ? expf(v[i] - m) : 0.f;
    z += v[i];
  }
  z = warp_sum(z);
#pragma unroll
  for (int i = 0; i < MAXE; ++i) v[i] = (lane + 32 * i < E) ? v[i] / z : -1.f;
  for (int r = 0; r < k; ++r) {
    float bv = -1.f;
    int bi = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < MAXE; ++i) {
      const int e = lane + 32 * i;
      if (v[i] > bv) { bv = v[i]; bi = e; }      // increasing e: ties keep the lower id
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
    }
    if (lane == 0) { ids[r] = bi; wts[r] = bv; }
#pragma unroll
    for (int i = 0; i < MAXE; ++i)
      if (lane + 32 * i == bi) v[i] = -1.f;        // taken
  }
}

// Where a permutation is written: the active-expert list (expert, offset into
// perm, pair count per slot), its length, and the pair permutation.
struct RouteOut {
  int* ex;
  int* off;
  int* cnt;
  int* n_active;
  int* perm;
};

// Per-expert pair lists and the active list from the ids [T, k] (block-wide).
// Slots 0..S-1 are the shared experts with every row (pairs r*NS + k + s),
// then the routed experts that have rows, in id order, each with its pairs in
// (row, slot) order. s_ids: the ids in shared memory; smi: shared scratch of
// 2*max(E,1) ints. Ends with a block barrier.
__device__ __forceinline__ void router_permute(const Dims& D, int T, const int* s_ids, int* smi,
                                               const RouteOut& O) {
  const int nk = T * D.k;
  int* cnt = smi;
  int* offs = cnt + (D.E > 0 ? D.E : 1);
  for (int e = threadIdx.x; e < D.E; e += blockDim.x) {
    int c = 0;
    for (int j = 0; j < nk; ++j) c += (s_ids[j] == e);
    cnt[e] = c;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int na = 0;
    for (int s = 0; s < D.S; ++s) {
      O.ex[na] = D.E + s; O.off[na] = s * T; O.cnt[na] = T;
      ++na;
    }
    int o = D.S * T;
    for (int e = 0; e < D.E; ++e) {
      offs[e] = o;
      if (cnt[e] > 0) {
        O.ex[na] = e; O.off[na] = o; O.cnt[na] = cnt[e];
        ++na;
      }
      o += cnt[e];
    }
    *O.n_active = na;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < D.S * T; i += blockDim.x) {
    const int s = i / T, r = i % T;
    O.perm[i] = r * D.NS + D.k + s;
  }
  for (int e = threadIdx.x; e < D.E; e += blockDim.x) {
    if (cnt[e] == 0) continue;
    int c = offs[e];
    for (int j = 0; j < nk; ++j)
      if (s_ids[j] == e) O.perm[c++] = (j / D.k) * D.NS + (j % D.k);
  }
  __syncthreads();
}


}  // namespace spec
