// Kernel-level entry point: rejection-sampling verification of K drafts per
// sequence against materialised target logits -- the stochastic counterpart
// of the greedy acceptance rule ("End-to-end OCR expert model architecture
// and acceleration principles", section 6.1 and section 11 item 2: rejection
// sampling keeps the output distribution equal to the target model's own).
//
// Rule (the published speculative-sampling rule, which has that property):
// with p_j = softmax(logits row j-1 / temperature) and the drafter's q_j,
// accept d_j while u_accept[j] * q_j(d_j) < p_j(d_j); at the first rejection
// draw the appended token from max(0, p_j - q_j) (normalised), else draw the
// bonus from p_(K+1). A draw is the inverse CDF in index order: the smallest v
// whose running sum of weights exceeds u_sample * (sum of all weights).
//
// One 512-thread block per sequence, everything in fp32 with fixed reduction
// orders (the result is a function of the sequence's own inputs):
//  * (max, sum of exp) of a row: each thread runs an online max/sum over the
//    float4 groups t, t + 512, ... in order, then a fixed xor-shuffle tree and
//    warp order combine the threads;
//  * a draw: the row is cut into tiles of 2,048 values; a tile's weights are
//    summed by a fixed scan (4 values per thread in order, warp shuffle scans
//    of 16 sub-blocks, sub-block totals in order) -- by one warp per tile for
//    the totals, by the whole block for the tile where the running sum (tile
//    order) passes the target, with the same arithmetic, to find the token.
#include <cuda_runtime.h>

#include "../../include/spec.h"
#include "kernels.h"

namespace spec {
namespace {

constexpr int RS_THREADS = 512;
constexpr int RS_WARPS = RS_THREADS / 32;
constexpr int RS_TILE = RS_THREADS * 4;
constexpr int RS_MAX_TILES = 128;                 // vocabularies up to 262,144
constexpr int RS_UNROLL = 8;                      // float4 loads in flight per thread

struct RsShared {
  float wm[RS_WARPS], ws[RS_WARPS];               // per-warp (max, sum)
  float wscan[RS_WARPS];                          // per-warp totals of a tile scan
  float tile_tot[RS_MAX_TILES];
  float m, z;
  int pick;
};

__device__ __forceinline__ void online_add(float& m, float& s, float x) {
  if (x > m) {
    s = s * expf(m - x) + 1.f;
    m = x;
  } else {
    s += expf(x - m);
  }
}
__device__ __forceinline__ void online_merge(float& m, float& s, float m2, float s2) {
  if (m2 == -INFINITY) return;
  if (m == -INFINITY) { m = m2; s = s2; return; }
  const float mm = fmaxf(m, m2);
  s = s * expf(m - mm) + s2 * expf(m2 - mm);
  m = mm;
}

// (max, sum of exp(x - max)) of x = row * inv_temp over the whole row, into sh.m / sh.z.
__device__ void row_stats(const float* __restrict__ row, int V, float inv_temp, RsShared& sh) {
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  const int n4 = V / 4;
  float m = -INFINITY, s = 0.f;
  for (int i0 = t; i0 < n4; i0 += RS_THREADS * RS_UNROLL) {
    float4 v[RS_UNROLL];
#pragma unroll
    for (int u = 0; u < RS_UNROLL; ++u) {
      const int i = i0 + u * RS_THREADS;
      v[u] = i < n4 ? __ldg(reinterpret_cast<const float4*>(row) + i)
                    : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    }
#pragma unroll
    for (int u = 0; u < RS_UNROLL; ++u) {
      if (i0 + u * RS_THREADS < n4) {
        online_add(m, s, v[u].x * inv_temp);
        online_add(m, s, v[u].y * inv_temp);
        online_add(m, s, v[u].z * inv_temp);
        online_add(m, s, v[u].w * inv_temp);
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o), s2 = __shfl_xor_sync(0xffffffffu, s, o);
    online_merge(m, s, m2, s2);
  }
  if (lane == 0) { sh.wm[w] = m; sh.ws[w] = s; }
  __syncthreads();
  if (t == 0) {
    float M = sh.wm[0], Z = sh.ws[0];
    for (int i = 1; i < RS_WARPS; ++i) online_merge(M, Z, sh.wm[i], sh.ws[i]);
    sh.m = M;
    sh.z = Z;
  }
  __syncthreads();
}

// Weights of the draw: p(v) - q(v) clamped at 0 (q: the drafter row, a
// one-hot at d when qrow is null and use_q, nothing when !use_q).
struct DrawRow {
  const float* row;
  const float* qrow;
  int d;
  bool use_q;
  float m, inv_z, inv_temp;
  __device__ float w(int v) const {
    const float p = expf(row[v] * inv_temp - m) * inv_z;
    if (!use_q) return p;
    const float q = qrow ? qrow[v] : (v == d ? 1.f : 0.f);
    return fmaxf(p - q, 0.f);
  }
};

// Block scan of tile `tile`: this thread's 4 weights and its exclusive prefix
// inside the tile; returns the tile total (the same value in every thread).
__device__ float tile_scan(const DrawRow& r, int V, int tile, float (&wv)[4], float& excl, RsShared& sh) {
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  const int v0 = tile * RS_TILE + 4 * t;
  float own = 0.f;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    wv[e] = v0 + e < V ? r.w(v0 + e) : 0.f;
    own += wv[e];
  }
  float inc = own;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += y;
  }
  if (lane == 31) sh.wscan[w] = inc;
  __syncthreads();
  float before = 0.f, total = 0.f;
  for (int i = 0; i < RS_WARPS; ++i) {
    if (i < w) before += sh.wscan[i];
    total += sh.wscan[i];
  }
  excl = before + inc - own;
  __syncthreads();                                 // wscan is reused by the next scan
  return total;
}

// The total tile_scan returns for `tile`, computed by one warp alone with the
// same arithmetic: sub-block w (the block scan's warp w) is this warp's
// inclusive shuffle scan of its lanes' 4-value sums, read at lane 31, and the
// sub-block totals are added in order.
__device__ float tile_total_warp(const DrawRow& r, int V, int tile) {
  const int lane = threadIdx.x & 31;
  float total = 0.f;
#pragma unroll 4
  for (int sub = 0; sub < RS_WARPS; ++sub) {
    const int v0 = tile * RS_TILE + 4 * (sub * 32 + lane);
    float own = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) own += v0 + e < V ? r.w(v0 + e) : 0.f;
    float inc = own;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += y;
    }
    total += __shfl_sync(0xffffffffu, inc, 31);
  }
  return total;
}

// Inverse-CDF draw over the weights of r with uniform u; -1 when every
// weight is zero. Every thread takes the same branches (the tile totals are
// read from shared memory after a barrier).
__device__ int draw(const DrawRow& r, int V, float u, RsShared& sh) {
  const int ntiles = (V + RS_TILE - 1) / RS_TILE;
  float wv[4], excl;
  for (int i = threadIdx.x >> 5; i < ntiles; i += RS_WARPS) {   // warps split the tiles, no barriers
    const float tot = tile_total_warp(r, V, i);
    if ((threadIdx.x & 31) == 0) sh.tile_tot[i] = tot;
  }
  __syncthreads();
  float S = 0.f;
  for (int i = 0; i < ntiles; ++i) S += sh.tile_tot[i];
  if (!(S > 0.f)) return -1;
  // the tile where the running sum (tile order) passes u * S
  const float target = u * S;
  int tile = -1;
  float base = 0.f, run = 0.f;
  for (int i = 0; i < ntiles; ++i) {
    if (run + sh.tile_tot[i] > target) { tile = i; base = run; break; }
    run += sh.tile_tot[i];
  }
  const bool last_positive = tile < 0;             // rounding put u * S at S: take the last positive weight
  if (last_positive) {
    for (int i = ntiles - 1; i >= 0; --i)
      if (sh.tile_tot[i] > 0.f) { tile = i; break; }
  }
  if (threadIdx.x == 0) sh.pick = 0x7fffffff;
  tile_scan(r, V, tile, wv, excl, sh);             // its barriers also publish sh.pick
  const int v0 = tile * RS_TILE + 4 * threadIdx.x;
  if (!last_positive) {
    // the smallest v of the tile whose running sum (tile base, exclusive
    // prefix, then this thread's values in order) passes the target
    float c = base + excl;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      c += wv[e];
      if (c > target && wv[e] > 0.f) {
        atomicMin(&sh.pick, v0 + e);
        break;
      }
    }
  }
  __syncthreads();
  int v = sh.pick;
  __syncthreads();
  if (v == 0x7fffffff) {
    // none passed it (rounding between the tile total and the running sums,
    // or u * S rounded to S): the last positive weight of the tile, which
    // exists because the tile's total is positive
    if (threadIdx.x == 0) sh.pick = -1;
    __syncthreads();
#pragma unroll
    for (int e = 3; e >= 0; --e)
      if (wv[e] > 0.f) { atomicMax(&sh.pick, v0 + e); break; }
    __syncthreads();
    v = sh.pick;
    __syncthreads();
  }
  return v;
}

__global__ void __launch_bounds__(RS_THREADS) k_rejection_sample(const float* __restrict__ logits,
                                                                 const int32_t* __restrict__ drafts,
                                                                 const float* __restrict__ q,
                                                                 const float* __restrict__ u_accept,
                                                                 const float* __restrict__ u_sample, int K, int V,
                                                                 float inv_temp, int32_t* out_acc, int32_t* out_tok) {
  __shared__ RsShared sh;
  const int s = blockIdx.x;
  for (int j = 0; j <= K; ++j) {
    const float* row = logits + ((size_t)s * (K + 1) + j) * V;
    row_stats(row, V, inv_temp, sh);
    DrawRow r{row, nullptr, -1, false, sh.m, 1.f / sh.z, inv_temp};
    if (j == K) {                                  // every draft accepted: the bonus from p_(K+1)
      const int t = draw(r, V, u_sample[(size_t)s * (K + 1) + K], sh);
      if (threadIdx.x == 0) { out_acc[s] = K; out_tok[s] = t; }
      return;
    }
    const int d = drafts[(size_t)s * K + j];
    if (d < 0 || d >= V) {                         // not a token: reported, nothing drawn
      if (threadIdx.x == 0) { out_acc[s] = -1; out_tok[s] = -1; }
      return;
    }
    const float* qrow = q ? q + ((size_t)s * K + j) * V : nullptr;
    const float pd = expf(row[d] * inv_temp - sh.m) * r.inv_z;
    const float qd = qrow ? qrow[d] : 1.f;
    if (u_accept[(size_t)s * K + j] * qd < pd) continue;
    // first rejection: the residual max(0, p - q); p == q everywhere leaves no
    // residual (a rejection then has probability zero) and p itself is drawn
    r.qrow = qrow;
    r.d = d;
    r.use_q = true;
    const float u = u_sample[(size_t)s * (K + 1) + j];
    int t = draw(r, V, u, sh);
    if (t < 0) {
      r.use_q = false;
      t = draw(r, V, u, sh);
    }
    if (threadIdx.x == 0) { out_acc[s] = j; out_tok[s] = t; }
    return;
  }
}

}  // namespace
}  // namespace spec

using namespace spec;

extern "C" int spec_rejection_sample(const float* logits_dev, const int32_t* drafts_dev, const float* q_dev,
                                     const float* u_accept_dev, const float* u_sample_dev, int n_seq, int K,
                                     int vocab, float temperature, int32_t* out_accepted_dev,
                                     int32_t* out_token_dev, uintptr_t cuda_stream) {
  if (!logits_dev || !u_sample_dev || !out_accepted_dev || !out_token_dev || (K > 0 && (!drafts_dev || !u_accept_dev)))
    return set_last_error(SPEC_ERR_ARG, "null pointer argument");
  if (n_seq < 1 || K < 0 || vocab < 4) return set_last_error(SPEC_ERR_ARG, "n_seq >= 1, K >= 0 and vocab >= 4 required");
  if (!(temperature > 0.f)) return set_last_error(SPEC_ERR_ARG, "temperature must be positive");
  if (vocab % 4 || vocab > RS_TILE * RS_MAX_TILES)
    return set_last_error(SPEC_ERR_UNSUPPORTED, "vocab must be a multiple of 4 and at most 262144");
  if (reinterpret_cast<uintptr_t>(logits_dev) % 16)
    return set_last_error(SPEC_ERR_ARG, "logits must be 16-byte aligned");
  k_rejection_sample<<<n_seq, RS_THREADS, 0, reinterpret_cast<cudaStream_t>(cuda_stream)>>>(
      logits_dev, drafts_dev, q_dev, u_accept_dev, u_sample_dev, K, vocab, 1.f / temperature, out_accepted_dev,
      out_token_dev);
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? SPEC_OK : set_last_error(SPEC_ERR_CUDA, cudaGetErrorString(e));
}
