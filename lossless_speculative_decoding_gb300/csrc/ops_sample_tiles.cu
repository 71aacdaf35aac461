// Sampled verify step on the tensor-core path: rejection sampling from the
// LM head's per-tile softmax statistics (the TC_STATS epilogue), the rule of
// the one-block and cooperative forms ("End-to-end OCR expert model
// architecture and acceleration principles", section 6.1 and section 11 item
// 2: rejection sampling keeps the output distribution equal to the target
// model's own), with the drafter certain of its drafts.
#include <cuda_runtime.h>

#include "common.cuh"

namespace spec {
namespace {

__device__ __forceinline__ void online_merge(float& m, float& s, float m2, float s2) {
  if (m2 == -INFINITY) return;
  if (m == -INFINITY) { m = m2; s = s2; return; }
  const float mm = fmaxf(m, m2);
  s = s * expf(m - mm) + s2 * expf(m2 - mm);
  m = mm;
}

// ---- sampled verify step over LM-head tile statistics (k_rs_tiles) -----------
// The LM head of a sampled step leaves, per (row, 128-row vocabulary tile),
// the tile's (m_t, s_t, s_t without the row's draft) of logit * it and the
// draft's logit (the TC_STATS epilogue). One block per sequence:
//  * a row's (max, sum): thread i merges tiles i, i + 256, ... in order, then
//    a fixed warp tree and warp order;
//  * the walk takes each acceptance decision from the draft's logit;
//  * the draw turns every tile's statistics into its total s_t exp(m_t - m) / z
//    (the draft's tile without the draft for the residual of a drafter certain
//    of its drafts), picks the tile where the running sum passes u * S (lanes
//    of warp 0 over contiguous tile ranges), recomputes that tile's 128 logits
//    from the row's LM-head input (the normed final state as its bf16 hi + lo
//    parts) and the tiled LM head, and scans them for the token.
// The recomputed logits sum in another order than the tensor cores, so a
// draw whose target lies within rounding of a bucket edge can differ.
constexpr int RT_THREADS = 256, RT_WARPS = RT_THREADS / 32, RT_TILE = 128;
constexpr int RT_MAX_H = 2560;                   // LM-head input width at most (8-value pieces per lane: 10)
constexpr int RT_MAX_TILES = 2048;               // vocabularies up to 262,144

struct RtShared {
  float T[RT_MAX_TILES];                         // tile totals of the draw
  float lg[RT_TILE];                             // the picked tile's logits
  float wsum[RT_WARPS];
  float2 red[RT_WARPS];
  float m, z, base, target;
  int tile, last_positive, pick;
};

// (max, sum) of a row from its tile statistics, in every thread.
__device__ float2 rt_merge(const float4* __restrict__ st, int NT, RtShared& sh) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  float m = -INFINITY, s = 0.f;
  for (int k = threadIdx.x; k < NT; k += RT_THREADS) {
    const float4 v = __ldcg(st + k);
    online_merge(m, s, v.x, v.y);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o), s2 = __shfl_xor_sync(0xffffffffu, s, o);
    online_merge(m, s, m2, s2);
  }
  if (lane == 0) sh.red[w] = make_float2(m, s);
  __syncthreads();
  if (threadIdx.x == 0) {
    float M = sh.red[0].x, Z = sh.red[0].y;
    for (int i = 1; i < RT_WARPS; ++i) online_merge(M, Z, sh.red[i].x, sh.red[i].y);
    sh.m = M;
    sh.z = Z;
  }
  __syncthreads();
  return make_float2(sh.m, sh.z);
}

// Draw over the tile totals in sh.T; the picked tile's logits are recomputed.
// Returns -1 when every total is zero.
__device__ int rt_draw(int NT, const uint16_t* __restrict__ W,
                       const uint16_t* __restrict__ xh, const uint16_t* __restrict__ xl, int h, float m, float inv_z,
                       float it, int d, bool residual, float u, RtShared& sh) {
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  if (w == 0) {
    const int per = (NT + 31) / 32, k0 = lane * per;
    float own = 0.f;
    for (int k = k0; k < min(NT, k0 + per); ++k) own += sh.T[k];
    float inc = own;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += y;
    }
    const float S = __shfl_sync(0xffffffffu, inc, 31);
    const float target = u * S;
    const unsigned pass = __ballot_sync(0xffffffffu, inc > target);
    const unsigned pos = __ballot_sync(0xffffffffu, own > 0.f);
    const int f = pass ? __ffs(pass) - 1 : (pos ? 31 - __clz(pos) : -1);
    if (lane == 0) { sh.tile = -1; sh.last_positive = 1; sh.target = target; sh.pick = 0x7fffffff; }
    __syncwarp();
    if (S > 0.f && lane == f) {
      float run = inc - own, base = 0.f;
      int tile = -1;
      bool found = false;
      for (int k = k0; k < min(NT, k0 + per); ++k) {
        if (pass && run + sh.T[k] > target) { tile = k; base = run; found = true; break; }
        if (sh.T[k] > 0.f) { tile = k; base = run; }
        run += sh.T[k];
      }
      sh.last_positive = !found;
      sh.tile = tile;
      sh.base = base;
    }
  }
  __syncthreads();
  const int tile = sh.tile;
  if (tile < 0) return -1;
  // the tile's 128 logits: warp w takes rows w, w + 8, ...; lane l the 8-value
  // pieces l, l + 32, ... of K (tiled layout: 64-wide K atoms of 128 rows,
  // row r's piece c at r * 64 + (c ^ (r % 8)) * 8 elements). The lane's input
  // values (hi + lo) are loaded once; a row's weight pieces are all in flight
  // before the first product.
  const int KT = h / 64, np = h / 8;
  float xin[RT_MAX_H / 256][8];
#pragma unroll
  for (int i = 0; i < RT_MAX_H / 256; ++i) {
    const int p = lane + 32 * i;
    if (p < np) {
      const uint4 hv = __ldg(reinterpret_cast<const uint4*>(xh + (size_t)p * 8));
      const uint4 lv = __ldg(reinterpret_cast<const uint4*>(xl + (size_t)p * 8));
      const uint32_t hh[4] = {hv.x, hv.y, hv.z, hv.w}, ll[4] = {lv.x, lv.y, lv.z, lv.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        xin[i][2 * q] = bf16_to_f((uint16_t)(hh[q] & 0xFFFF)) + bf16_to_f((uint16_t)(ll[q] & 0xFFFF));
        xin[i][2 * q + 1] = bf16_to_f((uint16_t)(hh[q] >> 16)) + bf16_to_f((uint16_t)(ll[q] >> 16));
      }
    }
  }
  for (int r = w; r < RT_TILE; r += RT_WARPS) {
    uint4 wv[RT_MAX_H / 256];
#pragma unroll
    for (int i = 0; i < RT_MAX_H / 256; ++i) {
      const int p = lane + 32 * i;
      if (p < np)
        wv[i] = __ldg(reinterpret_cast<const uint4*>(
            W + ((size_t)tile * KT + p / 8) * (RT_TILE * 64) + (size_t)r * 64 + (size_t)(((p % 8) ^ (r & 7)) * 8)));
    }
    float acc = 0.f;
#pragma unroll
    for (int i = 0; i < RT_MAX_H / 256; ++i) {
      if (lane + 32 * i >= np) continue;
      const uint32_t ww[4] = {wv[i].x, wv[i].y, wv[i].z, wv[i].w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        acc = fmaf(bf16_to_f((uint16_t)(ww[q] & 0xFFFF)), xin[i][2 * q], acc);
        acc = fmaf(bf16_to_f((uint16_t)(ww[q] >> 16)), xin[i][2 * q + 1], acc);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) sh.lg[r] = acc;
  }
  __syncthreads();
  // scan of the tile's weights: threads 0..127, one value each
  float wv = 0.f, inc = 0.f;
  const int v = tile * RT_TILE + t;
  if (t < RT_TILE) {
    const float p = expf(sh.lg[t] * it - m) * inv_z;
    wv = residual ? (v == d ? 0.f : p) : p;     // max(0, p - q) with q one-hot at d
    inc = wv;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += y;
    }
    if (lane == 31) sh.wsum[w] = inc;
  }
  __syncthreads();
  if (t < RT_TILE && !sh.last_positive) {
    float before = 0.f;
    for (int i = 0; i < w; ++i) before += sh.wsum[i];
    if (sh.base + before + inc > sh.target && wv > 0.f) atomicMin(&sh.pick, v);
  }
  __syncthreads();
  int pick = sh.pick;
  __syncthreads();
  if (pick == 0x7fffffff) {                       // the tile's last positive weight
    if (t == 0) sh.pick = -1;
    __syncthreads();
    if (t < RT_TILE && wv > 0.f) atomicMax(&sh.pick, v);
    __syncthreads();
    pick = sh.pick;
    __syncthreads();
  }
  return pick;
}

__global__ void __launch_bounds__(RT_THREADS, 1) k_rs_tiles(const float4* __restrict__ stats, const float* __restrict__ xd,
                                                         int NT, const uint16_t* __restrict__ W,
                                                         const uint16_t* __restrict__ xn_hi,
                                                         const uint16_t* __restrict__ xn_lo, int h,
                                                         const int32_t* __restrict__ drafts,
                                                         const int32_t* __restrict__ n_draft,
                                                         const float* __restrict__ u_accept,
                                                         const float* __restrict__ u_sample, const float* __restrict__ it_dev,
                                                         int K, int32_t* out_acc, int32_t* out_tok) {
  __shared__ RtShared sh;
  pdl_wait();
  const int s = blockIdx.x, lane = threadIdx.x & 31, R = K + 1;
  const float it = *it_dev;
  const int Ks = n_draft ? min(max(n_draft[s], 0), K) : K;
  const int V = NT * RT_TILE;
  int jinv = Ks;
  for (int c = 0; c < Ks && jinv == Ks; c += 32) {
    const int j = c + lane;
    const int dj = j < Ks ? drafts[(size_t)s * K + j] : 0;
    const unsigned bad = __ballot_sync(0xffffffffu, j < Ks && (dj < 0 || dj >= V));
    if (bad) jinv = c + __ffs(bad) - 1;
  }
  const int nr = jinv < Ks ? jinv : Ks + 1;
  int jrow = -1, d = -1;
  bool residual = false;
  float m = 0.f, inv_z = 0.f;
  for (int j = 0; j < nr; ++j) {
    const int t = s * R + j;
    const float2 mz = rt_merge(stats + (size_t)t * NT, NT, sh);
    const float iz = 1.f / mz.y;
    if (j == Ks) { jrow = j; m = mz.x; inv_z = iz; break; }          // every draft accepted: the bonus
    const float pd = expf(xd[t] * it - mz.x) * iz;
    if (u_accept[(size_t)s * K + j] < pd) continue;                  // q(d) = 1
    jrow = j; m = mz.x; inv_z = iz; d = drafts[(size_t)s * K + j]; residual = true;
    break;
  }
  int acc = -1, tok = -1;
  if (jrow >= 0) {
    const int t = s * R + jrow;
    const float4* st = stats + (size_t)t * NT;
    const float u = u_sample[(size_t)s * R + jrow];
    const uint16_t* xh = xn_hi + (size_t)t * h;
    const uint16_t* xl = xn_lo + (size_t)t * h;
    for (int pass = 0; pass < 2 && tok < 0; ++pass) {
      // the second pass (residual zero everywhere: a rejection then has
      // probability zero) draws from p itself
      const bool res = residual && pass == 0;
      const int dt = res ? d / RT_TILE : -1;
      for (int k = threadIdx.x; k < NT; k += RT_THREADS) {
        const float4 v = __ldcg(st + k);
        sh.T[k] = v.x == -INFINITY ? 0.f : (k == dt ? v.z : v.y) * expf(v.x - m) * inv_z;
      }
      __syncthreads();
      tok = rt_draw(NT, W, xh, xl, h, m, inv_z, it, d, res, u, sh);
      if (!residual) break;
    }
    acc = jrow;
  }
  if (threadIdx.x == 0) { out_acc[s] = acc; out_tok[s] = tok; }
}

}  // namespace

int rs_tiles_max_h() { return RT_MAX_H; }

void launch_rs_tiles(const float* stats, const float* xd, int V, const uint16_t* lm_head_tiled, const uint16_t* xn_hi,
                     const uint16_t* xn_lo, int h, const int32_t* drafts, const int32_t* n_draft, const float* u_accept,
                     const float* u_sample, const float* it_dev, int n_seq, int K, int32_t* out_acc, int32_t* out_tok,
                     cudaStream_t st) {
  launch_k(k_rs_tiles, dim3(n_seq), dim3(RT_THREADS), 0, st, reinterpret_cast<const float4*>(stats), xd, V / RT_TILE,
           lm_head_tiled, xn_hi, xn_lo, h, drafts, n_draft, u_accept, u_sample, it_dev, K, out_acc, out_tok);
}

}  // namespace spec
