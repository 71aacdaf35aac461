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
  for (int i = 0; i < MAXE; ++i) {
    const float p = v[i] / z;                     // a NaN probability ranks as 0, so ids stay < E
    v[i] = (lane + 32 * i < E) ? (p == p ? p : 0.f) : -1.f;
  }
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

// Shared scratch (ints) router_permute needs for nk = T * k routed pairs.
__host__ __device__ inline int permute_scratch_words(int E, int nk) {
  const int E1 = E > 0 ? E : 1;
  return 2 * E1 + ((nk + 31) / 32) * E1;
}

// Per-expert pair lists and the active list from the ids [T, k] (block-wide).
// Slots 0..S-1 are the shared experts with every row (pairs r*NS + k + s),
// then the routed experts that have rows, in id order, each with its pairs in
// increasing pair order j = r*k + slot. The pairs are cut into 32-pair chunks,
// one warp per chunk: __match_any_sync groups the lanes with the same expert,
// giving per-chunk counts and each pair's rank among the equal lanes before
// it; an exclusive prefix over chunks per expert and a warp scan over experts
// place every pair. s_ids: the ids in shared memory; smi: shared scratch of
// permute_scratch_words(E, T*k) ints. Ends with a block barrier.
__device__ __forceinline__ void router_permute(const Dims& D, int T, const int* s_ids, int* smi,
                                               const RouteOut& O) {
  const int nk = T * D.k;
  const int E1 = D.E > 0 ? D.E : 1;
  const int nchunk = (nk + 31) / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  int* cnt = smi;                 // [E] pairs per expert
  int* offs = cnt + E1;           // [E] first perm index of the expert
  int* pre = offs + E1;           // [nchunk][E] pairs of the expert in earlier chunks
  for (int i = threadIdx.x; i < nchunk * E1; i += blockDim.x) pre[i] = 0;
  __syncthreads();
  for (int w = warp; w < nchunk; w += nw) {
    const int j = w * 32 + lane;
    const int id = j < nk ? s_ids[j] : -1;
    const unsigned m = __match_any_sync(0xffffffffu, id);
    if (id >= 0 && lane == __ffs(m) - 1) pre[w * E1 + id] = __popc(m);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < D.E; e += blockDim.x) {
    int run = 0;
    for (int w = 0; w < nchunk; ++w) {
      const int c = pre[w * E1 + e];
      pre[w * E1 + e] = run;
      run += c;
    }
    cnt[e] = run;
  }
  __syncthreads();
  if (warp == 0) {
    // lane l owns experts [l*per, (l+1)*per): exclusive scans of pair counts
    // and of active experts give each expert its offset and active slot
    const int per = (D.E + 31) / 32, e0 = lane * per;
    int csum = 0, asum = 0;
    for (int i = 0; i < per; ++i) {
      const int e = e0 + i;
      if (e < D.E) { csum += cnt[e]; asum += cnt[e] > 0; }
    }
    int cx = csum, ax = asum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int c2 = __shfl_up_sync(0xffffffffu, cx, o), a2 = __shfl_up_sync(0xffffffffu, ax, o);
      if (lane >= o) { cx += c2; ax += a2; }
    }
    int off = D.S * T + cx - csum, na = D.S + ax - asum;
    for (int i = 0; i < per; ++i) {
      const int e = e0 + i;
      if (e < D.E) {
        offs[e] = off;
        if (cnt[e] > 0) {
          O.ex[na] = e; O.off[na] = off; O.cnt[na] = cnt[e];
          ++na;
        }
        off += cnt[e];
      }
    }
    for (int s = lane; s < D.S; s += 32) {
      O.ex[s] = D.E + s; O.off[s] = s * T; O.cnt[s] = T;
    }
    if (lane == 31) *O.n_active = D.S + ax;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < D.S * T; i += blockDim.x) {
    const int s = i / T, r = i % T;
    O.perm[i] = r * D.NS + D.k + s;
  }
  for (int w = warp; w < nchunk; w += nw) {
    const int j = w * 32 + lane;
    const int id = j < nk ? s_ids[j] : -1;
    const unsigned m = __match_any_sync(0xffffffffu, id);
    if (id >= 0) {
      const int rank = __popc(m & ((1u << lane) - 1u));
      O.perm[offs[id] + pre[w * E1 + id] + rank] = (j / D.k) * D.NS + (j % D.k);
    }
  }
  __syncthreads();
}


}  // namespace spec
