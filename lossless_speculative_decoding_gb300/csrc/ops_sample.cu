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

#include <algorithm>
#include <mutex>

#include "../../include/spec.h"
#include "common.cuh"

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
  __device__ float w(int v) const { return w_of(v, row[v], qrow ? qrow[v] : 0.f); }
  // the weight of v given its logit x and (with qrow) its drafter probability qv
  __device__ float w_of(int v, float x, float qv) const {
    const float p = expf(x * inv_temp - m) * inv_z;
    if (!use_q) return p;
    const float q = qrow ? qv : (v == d ? 1.f : 0.f);
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
  constexpr int HS = RS_WARPS / 2;                 // sub-blocks whose values are loaded together
  float total = 0.f;
#pragma unroll
  for (int h0 = 0; h0 < RS_WARPS; h0 += HS) {
    float4 xv[HS], qv[HS];
#pragma unroll
    for (int i = 0; i < HS; ++i) {
      const int v0 = tile * RS_TILE + 4 * ((h0 + i) * 32 + lane);
      xv[i] = v0 < V ? __ldg(reinterpret_cast<const float4*>(r.row + v0)) : make_float4(0.f, 0.f, 0.f, 0.f);
      qv[i] = (v0 < V && r.use_q && r.qrow) ? __ldg(reinterpret_cast<const float4*>(r.qrow + v0))
                                            : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int i = 0; i < HS; ++i) {
      const int v0 = tile * RS_TILE + 4 * ((h0 + i) * 32 + lane);
      const float x4[4] = {xv[i].x, xv[i].y, xv[i].z, xv[i].w};
      const float q4[4] = {qv[i].x, qv[i].y, qv[i].z, qv[i].w};
      float own = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) own += v0 + e < V ? r.w_of(v0 + e, x4[e], q4[e]) : 0.f;
      float inc = own;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += y;
      }
      total += __shfl_sync(0xffffffffu, inc, 31);
    }
  }
  return total;
}

// Inverse-CDF draw over the weights of r with uniform u; -1 when every
// weight is zero. Every thread takes the same branches (the tile totals are
// read from shared memory after a barrier).
__device__ int draw_pick(const DrawRow& r, int V, float u, RsShared& sh);
__device__ int draw(const DrawRow& r, int V, float u, RsShared& sh) {
  const int ntiles = (V + RS_TILE - 1) / RS_TILE;
  for (int i = threadIdx.x >> 5; i < ntiles; i += RS_WARPS) {   // warps split the tiles, no barriers
    const float tot = tile_total_warp(r, V, i);
    if ((threadIdx.x & 31) == 0) sh.tile_tot[i] = tot;
  }
  __syncthreads();
  return draw_pick(r, V, u, sh);
}

// The draw from the tile totals in sh.tile_tot (published before the call).
__device__ int draw_pick(const DrawRow& r, int V, float u, RsShared& sh) {
  const int ntiles = (V + RS_TILE - 1) / RS_TILE;
  float wv[4], excl;
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

// ---- cooperative form (spec_rejection_sample_ws) -----------------------------
// B blocks of 256 threads per sequence, all resident at once (a cooperative
// launch). A row is cut into tiles of 1,024 values; a warp reduces a tile to
// (max, sum of exp(x - max)) by rc_tile_stats (hardware base-2 exponential,
// relative error ~1e-6), plus the same sum without the row's draft. The rows are read in phases: a phase
// covers a run of rows (the first phase `first_rows` of them, later phases
// the rest), the blocks split its (row, tile) items, meet at a counter of the
// sequence (a bounded wait), merge each row's tile statistics in one fixed
// order and walk the acceptance rule over the phase's rows; a phase is only
// run while the walk has not stopped, so rows are read speculatively only
// within a phase. For the draw, a tile's total is its sum scaled to the row,
// exp(m_t - m) / z (the draft's tile without the draft for the residual of a
// one-hot drafter, whose max(0, p - q) is p with the draft's weight removed);
// with a drafter distribution q every block first sums max(0, p - q) over its
// tiles of the row. Block 0 picks the tile where the running sum (tile order)
// passes u * S and scans it for the token with the weights of the one-block
// form.
constexpr int RC_THREADS = 256, RC_WARPS = RC_THREADS / 32;
constexpr int RC_TILE = 1024;                    // values per tile: 8 float4 per lane
constexpr int RC_MAX_TILES = 256;                // vocabularies up to 262,144
constexpr int RC_TILES_PER_LANE = RC_MAX_TILES / 32;
constexpr int RC_PHASE_ROWS = 32;                // rows of a phase at most: one per lane

struct RcShared {
  float T[RC_MAX_TILES];                         // tile totals of the draw
  float2 mz[RC_PHASE_ROWS];                      // (max, sum) of the phase's rows
  float wsum[RC_WARPS];
  float base, target;
  int tile, last_positive, pick, ok;
};

// 2^x by the hardware approximation (ex2.approx: relative error ~2^-22;
// flushes subnormal results to zero).
__device__ __forceinline__ float ex2_fast(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
constexpr float RC_LOG2E = 1.4426950408889634f;  // log2(e): e^y = 2^(y log2 e)

// Statistics of one tile of x * it (one warp): m = the tile's max of x * it,
// s = sum of exp(x * it - m), and the same sum without value `skip` (equal to
// s unless `skip` lies in the tile). The max comes first (lanes, then an xor
// tree), so every exponential is taken against it: exp(x * it - m) as
// 2^(x * it log2 e - m log2 e), one fused multiply-add and one ex2.approx
// (relative error ~1e-6 with the argument's rounding). The sums: the lane's
// 32 values in order, then an xor tree.
__device__ float3 rc_tile_stats(const float* __restrict__ row, int V, int tile, float it, int skip) {
  const int lane = threadIdx.x & 31, n4 = V / 4;
  float4 v[RC_TILE / 128];
#pragma unroll
  for (int i = 0; i < RC_TILE / 128; ++i) {
    const int i4 = tile * (RC_TILE / 4) + i * 32 + lane;
    v[i] = i4 < n4 ? __ldg(reinterpret_cast<const float4*>(row) + i4)
                   : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
  }
  float mx = -INFINITY;
#pragma unroll
  for (int i = 0; i < RC_TILE / 128; ++i) mx = fmaxf(mx, fmaxf(fmaxf(v[i].x, v[i].y), fmaxf(v[i].z, v[i].w)));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  const float m = mx * it;                       // rounding is monotone: the max of x * it
  if (m == -INFINITY) return make_float3(m, 0.f, 0.f);
  const float c = it * RC_LOG2E, mb = m * RC_LOG2E;
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < RC_TILE / 128; ++i)
    s += (ex2_fast(fmaf(v[i].x, c, -mb)) + ex2_fast(fmaf(v[i].y, c, -mb))) +
         (ex2_fast(fmaf(v[i].z, c, -mb)) + ex2_fast(fmaf(v[i].w, c, -mb)));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  float sk = s;
  if (skip >= tile * RC_TILE && skip < (tile + 1) * RC_TILE) {   // the same for every lane
    sk = 0.f;
#pragma unroll
    for (int i = 0; i < RC_TILE / 128; ++i) {
      const int k = skip - 4 * (tile * (RC_TILE / 4) + i * 32 + lane);   // the skipped value's place, if here
      const float e0 = k == 0 ? 0.f : ex2_fast(fmaf(v[i].x, c, -mb));
      const float e1 = k == 1 ? 0.f : ex2_fast(fmaf(v[i].y, c, -mb));
      const float e2 = k == 2 ? 0.f : ex2_fast(fmaf(v[i].z, c, -mb));
      const float e3 = k == 3 ? 0.f : ex2_fast(fmaf(v[i].w, c, -mb));
      sk += (e0 + e1) + (e2 + e3);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sk += __shfl_xor_sync(0xffffffffu, sk, o);
  }
  return make_float3(m, s, sk);
}

// (max, sum) of a row from its tile statistics, in every lane of the calling
// warp: lane l merges tiles l, l + 32, ... in that order, then a fixed tree.
__device__ float2 rc_merge(const float4* __restrict__ ts, int NT) {
  const int lane = threadIdx.x & 31;
  float4 st[RC_TILES_PER_LANE];
#pragma unroll
  for (int k = 0; k < RC_TILES_PER_LANE; ++k) {
    const int t = lane + 32 * k;
    st[k] = t < NT ? __ldcg(ts + t) : make_float4(-INFINITY, 0.f, 0.f, 0.f);
  }
  float m = -INFINITY, s = 0.f;
#pragma unroll
  for (int k = 0; k < RC_TILES_PER_LANE; ++k) online_merge(m, s, st[k].x, st[k].y);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o), s2 = __shfl_xor_sync(0xffffffffu, s, o);
    online_merge(m, s, m2, s2);
  }
  return make_float2(m, s);
}

// A tile's total from its statistics: the tile's sum (without the draft in
// the draft's tile, when d_tile names it) scaled to the row.
__device__ __forceinline__ float rc_total(const float4& st, int t, int d_tile, float m, float inv_z) {
  return st.x == -INFINITY ? 0.f : (t == d_tile ? st.z : st.y) * expf(st.x - m) * inv_z;
}

// The block's arrival at the sequence's counter, then (with `wait`) a wait
// until `target` arrivals in all. The barrier orders the block's writes
// before thread 0's release fence; the acquire fence after the wait orders
// the other blocks' writes before this block's reads. False when the wait
// ran past WAIT_DEADLINE_NS.
__device__ bool rc_sync(int* cnt, int target, bool wait, RcShared& sh) {
  __syncthreads();
  if (threadIdx.x == 0) {
    asm volatile("fence.acq_rel.gpu;" ::: "memory");
    asm volatile("red.relaxed.gpu.global.add.s32 [%0], 1;" ::"l"(cnt) : "memory");
    int ok = 1;
    if (wait) {
      auto arrived = [&]() {
        int v;
        asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(cnt) : "memory");
        return v >= target;
      };
      if (!arrived()) {
        const unsigned long long t0 = globaltimer_ns();
        while (!arrived())
          if (globaltimer_ns() - t0 > WAIT_DEADLINE_NS) { ok = 0; break; }
      }
      asm volatile("fence.acq_rel.gpu;" ::: "memory");
    }
    sh.ok = ok;
  }
  __syncthreads();
  return sh.ok != 0;
}

// The draw of block 0 from the tile totals in sh.T (the draw row's weights in
// r); -1 when every total is zero.
__device__ int rc_pick(const DrawRow& r, int V, int NT, float u, RcShared& sh) {
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  if (w == 0) {
    float own = 0.f;
#pragma unroll
    for (int k = 0; k < RC_TILES_PER_LANE; ++k) {
      const int i = lane * RC_TILES_PER_LANE + k;
      own += i < NT ? sh.T[i] : 0.f;
    }
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
    // the lane whose tiles hold the crossing; none (u * S rounded to S): the
    // last lane with a positive tile, whose last positive tile is taken
    const int f = pass ? __ffs(pass) - 1 : (pos ? 31 - __clz(pos) : -1);
    if (lane == 0) { sh.tile = -1; sh.last_positive = pass == 0; sh.target = target; }
    __syncwarp();
    if (S > 0.f && lane == f) {
      // the first of the lane's tiles where the running sum passes the target;
      // failing that (rounding), its last positive tile, taken at its last
      // positive weight
      float run = inc - own, base = 0.f;
      int tile = -1;
      bool found = false;
      for (int k = 0; k < RC_TILES_PER_LANE; ++k) {
        const int i = lane * RC_TILES_PER_LANE + k;
        if (i >= NT) break;
        if (pass && run + sh.T[i] > target) { tile = i; base = run; found = true; break; }
        if (sh.T[i] > 0.f) { tile = i; base = run; }
        run += sh.T[i];
      }
      sh.last_positive = !found;
      sh.tile = tile;
      sh.base = base;
    }
    if (lane == 0) sh.pick = 0x7fffffff;
  }
  __syncthreads();
  const int tile = sh.tile;
  if (tile < 0) return -1;
  // block scan of the tile: thread t holds values 4t .. 4t + 3
  const int v0 = tile * RC_TILE + 4 * t;
  float wv[4], own = 0.f;
  if (v0 < V) {
    const float4 x = __ldg(reinterpret_cast<const float4*>(r.row + v0));
    float4 qv = make_float4(0.f, 0.f, 0.f, 0.f);
    if (r.use_q && r.qrow) qv = __ldg(reinterpret_cast<const float4*>(r.qrow + v0));
    wv[0] = r.w_of(v0, x.x, qv.x);
    wv[1] = r.w_of(v0 + 1, x.y, qv.y);
    wv[2] = r.w_of(v0 + 2, x.z, qv.z);
    wv[3] = r.w_of(v0 + 3, x.w, qv.w);
  } else {
    wv[0] = wv[1] = wv[2] = wv[3] = 0.f;
  }
  own = (wv[0] + wv[1]) + (wv[2] + wv[3]);
  float inc = own;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += y;
  }
  if (lane == 31) sh.wsum[w] = inc;
  __syncthreads();
  float before = 0.f;
  for (int i = 0; i < w; ++i) before += sh.wsum[i];
  if (!sh.last_positive) {
    float c = sh.base + before + inc - own;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      c += wv[e];
      if (c > sh.target && wv[e] > 0.f) {
        atomicMin(&sh.pick, v0 + e);
        break;
      }
    }
  }
  __syncthreads();
  int v = sh.pick;
  __syncthreads();
  if (v == 0x7fffffff) {
    // none passed it (rounding between the tile total and the running sums):
    // the tile's last positive weight
    if (t == 0) sh.pick = -1;
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

// Tile totals of p_row in sh.T from the tile statistics (the draft's tile
// without the draft when d_tile names it); the whole block.
__device__ void rc_totals_from_stats(const float4* __restrict__ ts, int NT, float m, float inv_z, int d_tile,
                                     RcShared& sh) {
  for (int i = threadIdx.x; i < NT; i += RC_THREADS) sh.T[i] = rc_total(__ldcg(ts + i), i, d_tile, m, inv_z);
  __syncthreads();
}

// Counters of a sequence in the workspace: arrivals, then blocks done.
__global__ void __launch_bounds__(RC_THREADS, 4) k_rs_coop(
    const float* __restrict__ logits, const int32_t* __restrict__ drafts, const float* __restrict__ q,
    const float* __restrict__ u_accept, const float* __restrict__ u_sample, const int* __restrict__ n_draft,
    int n_seq, int K, int V, float it_arg, const float* __restrict__ it_dev, int B, int n_groups, int first_rows,
    int* __restrict__ ctr, float4* __restrict__ tstat, float* __restrict__ rtot, int32_t* out_acc,
    int32_t* out_tok) {
  __shared__ RcShared sh;
  const float it = it_dev ? *it_dev : it_arg;
  const int group = blockIdx.x / B, b = blockIdx.x % B, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int NT = (V + RC_TILE - 1) / RC_TILE;
  enum { INVALID, BONUS, RESIDUAL };
  auto row_of = [&](int s, int r) { return logits + ((size_t)s * (K + 1) + r) * V; };
  auto stats_of = [&](int s, int r) { return tstat + ((size_t)s * (K + 1) + r) * RC_MAX_TILES; };
  for (int s = group; s < n_seq; s += n_groups) {
    int* cnt = ctr + 2 * s;
    // this sequence's drafts: Ks of the K slots (its bonus row is row Ks)
    const int Ks = n_draft ? min(max(__ldg(n_draft + s), 0), K) : K;
    // the rows the walk can reach: a draft that is not a token ends it there
    int jinv = Ks;
    for (int c = 0; c < Ks && jinv == Ks; c += 32) {
      const int j = c + lane;
      const int dj = j < Ks ? __ldg(drafts + (size_t)s * K + j) : 0;
      const unsigned bad = __ballot_sync(0xffffffffu, j < Ks && (dj < 0 || dj >= V));
      if (bad) jinv = c + __ffs(bad) - 1;
    }
    const int nr = jinv < Ks ? jinv : Ks + 1;
    int kind = INVALID, jrow = -1, d = -1, phase = 0;
    bool decided = false, ok = true;
    float m = 0.f, inv_z = 0.f;
    for (int r0 = 0; r0 < nr && !decided; ++phase) {
      const int r1 = min(nr, r0 + (phase == 0 ? first_rows : RC_PHASE_ROWS));
      const int nrow = r1 - r0, items = nrow * NT;
      // lane l holds row r0 + l's draft and the inputs of its decision
      const int rl = r0 + lane;
      const bool dec_l = lane < nrow && rl < Ks;
      const int d_l = dec_l ? __ldg(drafts + (size_t)s * K + rl) : -1;
      const float xd_l = dec_l ? __ldg(row_of(s, rl) + d_l) : 0.f;
      const float qd_l = dec_l && q ? __ldg(q + ((size_t)s * K + rl) * V + d_l) : 1.f;
      const float ua_l = dec_l ? __ldg(u_accept + (size_t)s * K + rl) : 0.f;
      // this warp's (row, tile) items: i = i0, i0 + di, ...
      const int i0 = b * RC_WARPS + warp, di = RC_WARPS * B;
      for (int i = i0, rr = i0 / NT, t = i0 % NT; i < items; i += di) {
        const int dr = __shfl_sync(0xffffffffu, d_l, rr);
        const float3 st = rc_tile_stats(row_of(s, r0 + rr), V, t, it, dr);
        if (lane == 0) stats_of(s, r0 + rr)[t] = make_float4(st.x, st.y, st.z, 0.f);
        for (t += di; t >= NT; t -= NT) ++rr;        // the next item's (row, tile)
      }
      ok = rc_sync(cnt, B * (phase + 1), true, sh);
      if (!ok) break;
      // the phase's row statistics, a warp a row
      for (int rr = warp; rr < nrow; rr += RC_WARPS) {
        const float2 mz = rc_merge(stats_of(s, r0 + rr), NT);
        if (lane == 0) sh.mz[rr] = mz;
      }
      __syncthreads();
      // the walk over the phase's rows (every warp takes the same decisions)
      for (int rr = 0; rr < nrow; ++rr) {
        const float2 mz = sh.mz[rr];
        const float xd = __shfl_sync(0xffffffffu, xd_l, rr), qd = __shfl_sync(0xffffffffu, qd_l, rr);
        const float ua = __shfl_sync(0xffffffffu, ua_l, rr);
        const int dr = __shfl_sync(0xffffffffu, d_l, rr);
        const float iz = 1.f / mz.y;
        if (r0 + rr == Ks) {                           // every draft accepted: the bonus from p_(Ks+1)
          kind = BONUS;
        } else {
          if (ua * qd < expf(xd * it - mz.x) * iz) continue;
          kind = RESIDUAL;
          d = dr;
        }
        jrow = r0 + rr;
        m = mz.x;
        inv_z = iz;
        decided = true;
        break;
      }
      r0 = r1;
    }
    // not decided: every draft before the first non-token accepted (reported, nothing drawn)
    const float* row = jrow >= 0 ? row_of(s, jrow) : logits;
    const float* qrow = (kind == RESIDUAL && q) ? q + ((size_t)s * K + jrow) * V : nullptr;
    DrawRow r{row, qrow, d, kind == RESIDUAL, m, inv_z, it};
    if (ok && qrow) {
      // residual totals max(0, p - q) over this block's tiles of the row (one
      // warp a tile: the lane's values in order, then a fixed tree)
      for (int t = b * RC_WARPS + warp; t < NT; t += RC_WARPS * B) {
        float acc = 0.f;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          float4 xv[4], qv[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int i4 = t * (RC_TILE / 4) + (4 * h + i) * 32 + lane;
            xv[i] = i4 < V / 4 ? __ldg(reinterpret_cast<const float4*>(row) + i4) : make_float4(0.f, 0.f, 0.f, 0.f);
            qv[i] = i4 < V / 4 ? __ldg(reinterpret_cast<const float4*>(qrow) + i4) : make_float4(0.f, 0.f, 0.f, 0.f);
          }
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int v0 = 4 * (t * (RC_TILE / 4) + (4 * h + i) * 32 + lane);
            if (v0 >= V) continue;
            acc += (r.w_of(v0, xv[i].x, qv[i].x) + r.w_of(v0 + 1, xv[i].y, qv[i].y)) +
                   (r.w_of(v0 + 2, xv[i].z, qv[i].z) + r.w_of(v0 + 3, xv[i].w, qv[i].w));
          }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (lane == 0) rtot[(size_t)s * RC_MAX_TILES + t] = acc;
      }
      ok = rc_sync(cnt, B * (phase + 1), b == 0, sh);
    }
    if (b == 0) {
      int acc = -1, tok = -1;
      if (!ok) {
        acc = -2;                                    // a wait ran out
      } else if (kind != INVALID) {
        acc = jrow;
        if (qrow) {
          for (int i = threadIdx.x; i < NT; i += RC_THREADS) sh.T[i] = __ldcg(rtot + (size_t)s * RC_MAX_TILES + i);
          __syncthreads();
        } else {
          rc_totals_from_stats(stats_of(s, jrow), NT, m, inv_z, kind == RESIDUAL ? d / RC_TILE : -1, sh);
        }
        const float u = __ldg(u_sample + (size_t)s * (K + 1) + jrow);
        tok = rc_pick(r, V, NT, u, sh);
        if (tok < 0 && kind == RESIDUAL) {
          // p == q everywhere leaves no residual (a rejection then has
          // probability zero): p itself is drawn
          r.use_q = false;
          r.qrow = nullptr;
          rc_totals_from_stats(stats_of(s, jrow), NT, m, inv_z, -1, sh);
          tok = rc_pick(r, V, NT, u, sh);
        }
      }
      if (threadIdx.x == 0) { out_acc[s] = acc; out_tok[s] = tok; }
    }
    // the last block of the sequence to leave zeroes its counters: every
    // arrival of the sequence has happened by then
    __syncthreads();
    if (threadIdx.x == 0) {
      asm volatile("fence.acq_rel.gpu;" ::: "memory");
      if (atomicAdd(ctr + 2 * s + 1, 1) == B - 1) {
        atomicExch(ctr + 2 * s, 0);
        atomicExch(ctr + 2 * s + 1, 0);
      }
    }
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
  if (reinterpret_cast<uintptr_t>(logits_dev) % 16 || reinterpret_cast<uintptr_t>(q_dev) % 16)
    return set_last_error(SPEC_ERR_ARG, "logits and q must be 16-byte aligned");
  k_rejection_sample<<<n_seq, RS_THREADS, 0, reinterpret_cast<cudaStream_t>(cuda_stream)>>>(
      logits_dev, drafts_dev, q_dev, u_accept_dev, u_sample_dev, K, vocab, 1.f / temperature, out_accepted_dev,
      out_token_dev);
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? SPEC_OK : set_last_error(SPEC_ERR_CUDA, cudaGetErrorString(e));
}

// Workspace: per sequence two counters (arrivals, blocks done), then tile
// statistics [n_seq][K + 1][RC_MAX_TILES] float4, then residual tile totals
// [n_seq][RC_MAX_TILES] float.
static size_t rs_ws_layout(int n_seq, int K, size_t* off_ts, size_t* off_rt) {
  size_t o = ((size_t)n_seq * 2 * sizeof(int) + 15) & ~size_t(15);
  *off_ts = o;
  o += (size_t)n_seq * (K + 1) * RC_MAX_TILES * sizeof(float4);
  *off_rt = o;
  return o + (size_t)n_seq * RC_MAX_TILES * sizeof(float);
}

// Largest read of all K + 1 rows of all sequences done in one phase.
constexpr double RS_ONE_PHASE_BYTES = 24e6;

// Blocks of k_rs_coop that can be resident at once on the current device.
static int rs_coop_capacity() {
  static std::mutex mu;
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (cached[dev] == 0) {
    int per_sm = 0, sms = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_rs_coop, RC_THREADS, 0) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return 0;
    cached[dev] = per_sm * sms;
  }
  return cached[dev];
}

extern "C" int64_t spec_rejection_sample_ws_bytes(int n_seq, int K) {
  if (n_seq < 1 || K < 0) return set_last_error(SPEC_ERR_ARG, "n_seq >= 1 and K >= 0 required");
  size_t a, b;
  return (int64_t)rs_ws_layout(n_seq, K, &a, &b);
}

namespace spec {
int rs_coop_blocks() { return rs_coop_capacity(); }

size_t rs_coop_ws_bytes(int n_seq, int K) {
  size_t a, b;
  return rs_ws_layout(n_seq, K, &a, &b);
}

cudaError_t launch_rs_coop(const float* logits, const int32_t* drafts, const int32_t* n_draft, const float* q,
                           const float* u_accept, const float* u_sample, int n_seq, int K, int vocab, float it,
                           const float* it_dev, int32_t* out_acc, int32_t* out_tok, void* ws, cudaStream_t st) {
  const int cap = rs_coop_capacity();
  if (cap < 1) return cudaErrorCooperativeLaunchTooLarge;
  size_t off_ts, off_rt;
  rs_ws_layout(n_seq, K, &off_ts, &off_rt);
  // the first phase: every row when all of them are a small read (a few
  // microseconds of HBM time, less than the phases saved), else row 0 alone
  const int NT = (vocab + RC_TILE - 1) / RC_TILE;
  const double all_rows = (double)n_seq * (K + 1) * vocab * sizeof(float);
  const int first_rows = all_rows <= RS_ONE_PHASE_BYTES ? std::min(K + 1, RC_PHASE_ROWS) : 1;
  // B blocks per sequence (no more than the first phase has tiles for their
  // warps), as many sequences at once as fit; a block runs on over further
  // sequences
  const int B = std::max(1, std::min((first_rows * NT + RC_WARPS - 1) / RC_WARPS, cap / n_seq));
  const int n_groups = std::min(n_seq, cap / B);
  char* w = static_cast<char*>(ws);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n_groups * B);
  cfg.blockDim = dim3(RC_THREADS);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_rs_coop, logits, drafts, q, u_accept, u_sample, n_draft, n_seq, K, vocab, it,
                            it_dev, B, n_groups, first_rows, reinterpret_cast<int*>(w),
                            reinterpret_cast<float4*>(w + off_ts), reinterpret_cast<float*>(w + off_rt), out_acc,
                            out_tok);
}

// Stage a sampled step's uniforms and 1 / temperature into the model's buffer
// [u_accept (n_seq x K) | u_sample (n_seq x (K + 1)) | 1 / temperature].
__global__ void k_stage_sample(float* dst, int ua_cap, int us_cap, const float* ua, const float* us, int n_seq,
                               int K, float it) {
  for (int i = threadIdx.x; i < n_seq * K; i += blockDim.x) dst[i] = ua[i];
  for (int i = threadIdx.x; i < n_seq * (K + 1); i += blockDim.x) dst[ua_cap + i] = us[i];
  if (threadIdx.x == 0) dst[ua_cap + us_cap] = it;
}

void launch_stage_sample(float* dst, int max_batch, int K, const float* ua, const float* us, int n_seq, float it,
                         cudaStream_t st) {
  k_stage_sample<<<1, 256, 0, st>>>(dst, max_batch * K, max_batch * (K + 1), ua, us, n_seq, K, it);
}
}  // namespace spec

extern "C" int spec_rejection_sample_ws(const float* logits_dev, const int32_t* drafts_dev, const float* q_dev,
                                        const float* u_accept_dev, const float* u_sample_dev, int n_seq, int K,
                                        int vocab, float temperature, int32_t* out_accepted_dev,
                                        int32_t* out_token_dev, void* ws_dev, size_t ws_bytes,
                                        uintptr_t cuda_stream) {
  if (!logits_dev || !u_sample_dev || !out_accepted_dev || !out_token_dev || !ws_dev ||
      (K > 0 && (!drafts_dev || !u_accept_dev)))
    return set_last_error(SPEC_ERR_ARG, "null pointer argument");
  if (n_seq < 1 || K < 0 || vocab < 4) return set_last_error(SPEC_ERR_ARG, "n_seq >= 1, K >= 0 and vocab >= 4 required");
  if (!(temperature > 0.f)) return set_last_error(SPEC_ERR_ARG, "temperature must be positive");
  if (vocab % 4 || vocab > RC_TILE * RC_MAX_TILES)
    return set_last_error(SPEC_ERR_UNSUPPORTED, "vocab must be a multiple of 4 and at most 262144");
  if (reinterpret_cast<uintptr_t>(logits_dev) % 16 || reinterpret_cast<uintptr_t>(q_dev) % 16 ||
      reinterpret_cast<uintptr_t>(ws_dev) % 16)
    return set_last_error(SPEC_ERR_ARG, "logits, q and the workspace must be 16-byte aligned");
  if (ws_bytes < rs_coop_ws_bytes(n_seq, K)) return set_last_error(SPEC_ERR_ARG, "workspace too small");
  const cudaError_t e = launch_rs_coop(logits_dev, drafts_dev, nullptr, q_dev, u_accept_dev, u_sample_dev, n_seq, K,
                                       vocab, 1.f / temperature, nullptr, out_accepted_dev, out_token_dev, ws_dev,
                                       reinterpret_cast<cudaStream_t>(cuda_stream));
  return e == cudaSuccess ? SPEC_OK : set_last_error(SPEC_ERR_CUDA, cudaGetErrorString(e));
}
