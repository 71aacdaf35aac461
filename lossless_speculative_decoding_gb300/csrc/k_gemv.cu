// Weight-streaming GEMV kernels of the verify step.
//
// At verify-step sizes (a few rows per sequence) every projection reads each
// weight once and uses it for only T rows, so these kernels are bound by HBM
// bandwidth: each warp streams R = 4 weight rows with 16-byte non-allocating
// loads (GEMV_G chunks in flight per lane), multiplies them against up to
// TP = 4 activation rows staged in shared memory, and reduces the lane
// partials with a fixed butterfly. Every output element is computed in the
// same order whatever T, the row's place in the batch or the launch shape,
// which keeps speculative and plain greedy decoding bit-identical on the GPU
// (the lossless property of greedy verification: "Jina-OCR-v1", abstract).
//
// Fused epilogues: RMSNorm of the input rows in the prologue; RoPE and the
// paged KV write after the QKV projection; the residual add after the output
// projection; SwiGLU after the expert gate/up projection; a per-row argmax
// after the LM head so logits are never written (unless a debug buffer is
// given).
#include "common.cuh"
#include "kernels.h"

namespace spec {

// ---------------------------------------------------------------------------
// Warp reduce-scatter of N partial sums (N = 16 or 32): after it, the lane
// returns the full warp sum of value index (N == 32 ? lane : lane >> 1).
// The pairing tree is the same for every value index.
template <int N>
__device__ __forceinline__ float reduce_scatter(float (&a)[N]) {
  const int lane = threadIdx.x & 31;
  int n = N;
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) {
    if (n > 1) {
      const bool up = (lane & m) != 0;
#pragma unroll
      for (int i = 0; i < N / 2; ++i) {
        if (i < n / 2) {
          const float send = up ? a[i] : a[i + n / 2];
          const float keep = up ? a[i + n / 2] : a[i];
          a[i] = keep + __shfl_xor_sync(0xffffffffu, send, m);
        }
      }
      n >>= 1;
    } else {
      a[0] += __shfl_xor_sync(0xffffffffu, a[0], m);
    }
  }
  return a[0];
}

// Group q (of per16/4) of four elements of a 16-byte vector, as floats.
template <class WT, int Q> __device__ __forceinline__ void unpack4(const uint4& v, float* o);
template <> __device__ __forceinline__ void unpack4<float, 0>(const uint4& v, float* o) {
  o[0] = __uint_as_float(v.x); o[1] = __uint_as_float(v.y); o[2] = __uint_as_float(v.z); o[3] = __uint_as_float(v.w);
}
__device__ __forceinline__ void bf2(uint32_t w, float* o) {
  o[0] = __uint_as_float(w << 16); o[1] = __uint_as_float(w & 0xFFFF0000u);
}
template <> __device__ __forceinline__ void unpack4<bf16_t, 0>(const uint4& v, float* o) { bf2(v.x, o); bf2(v.y, o + 2); }
template <> __device__ __forceinline__ void unpack4<bf16_t, 1>(const uint4& v, float* o) { bf2(v.z, o); bf2(v.w, o + 2); }
__device__ __forceinline__ void f8x4(uint32_t w, float* o) {
  __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w & 0xFFFF), __NV_E4M3);
  __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w >> 16), __NV_E4M3);
  float2 a = __half22float2(*reinterpret_cast<__half2*>(&lo));
  float2 b = __half22float2(*reinterpret_cast<__half2*>(&hi));
  o[0] = a.x; o[1] = a.y; o[2] = b.x; o[3] = b.y;
}
template <> __device__ __forceinline__ void unpack4<fp8_t, 0>(const uint4& v, float* o) { f8x4(v.x, o); }
template <> __device__ __forceinline__ void unpack4<fp8_t, 1>(const uint4& v, float* o) { f8x4(v.y, o); }
template <> __device__ __forceinline__ void unpack4<fp8_t, 2>(const uint4& v, float* o) { f8x4(v.z, o); }
template <> __device__ __forceinline__ void unpack4<fp8_t, 3>(const uint4& v, float* o) { f8x4(v.w, o); }

template <class WT, int R, int TP, int Q>
__device__ __forceinline__ void fma_group(const uint4 (&wv)[R], const float* xs, int ldxs, int k,
                                          float (&acc)[R * TP]) {
  float xv[TP][4];
#pragma unroll
  for (int t = 0; t < TP; ++t) {
    const float4 x4 = *reinterpret_cast<const float4*>(xs + t * ldxs + k + 4 * Q);
    xv[t][0] = x4.x; xv[t][1] = x4.y; xv[t][2] = x4.z; xv[t][3] = x4.w;
  }
#pragma unroll
  for (int r = 0; r < R; ++r) {
    float w[4];
    unpack4<WT, Q>(wv[r], w);
#pragma unroll
    for (int t = 0; t < TP; ++t)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[r * TP + t] = fmaf(w[e], xv[t][e], acc[r * TP + t]);
  }
}

// acc[r*TP + t] = sum_k W[row r][k] * xs[t][k] over this lane's 16-byte chunks
// (chunk c = lane, lane + 32, ... in increasing order).
template <class WT, int R, int TP>
__device__ __forceinline__ void gemv_lane(const WT* const (&wrow)[R], int K, const float* xs, int ldxs,
                                          float (&acc)[R * TP]) {
  constexpr int EP = Elt<WT>::per16;
  const int nch = K / EP;
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int i = 0; i < R * TP; ++i) acc[i] = 0.f;
  for (int c0 = lane; c0 < nch; c0 += 32 * GEMV_G) {
    uint4 wv[GEMV_G][R];
#pragma unroll
    for (int g = 0; g < GEMV_G; ++g) {
      const int c = c0 + g * 32;
#pragma unroll
      for (int r = 0; r < R; ++r)
        wv[g][r] = (c < nch) ? ld_stream(wrow[r] + (size_t)c * EP) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int g = 0; g < GEMV_G; ++g) {
      const int c = c0 + g * 32;
      if (c < nch) {
        const int k = c * EP;
        fma_group<WT, R, TP, 0>(wv[g], xs, ldxs, k, acc);
        if constexpr (EP >= 8) fma_group<WT, R, TP, 1>(wv[g], xs, ldxs, k, acc);
        if constexpr (EP >= 16) {
          fma_group<WT, R, TP, 2>(wv[g], xs, ldxs, k, acc);
          fma_group<WT, R, TP, 3>(wv[g], xs, ldxs, k, acc);
        }
      }
    }
  }
}

// Stage TP activation rows into shared memory (zeros past `nvalid`).
// src_row(t) gives the source row pointer. With gamma != nullptr each row is
// RMS-normalised: x / sqrt(mean(x^2) + eps) * gamma (warp t sums row t).
template <class F>
__device__ __forceinline__ void stage_rows(float* xs, int K, int nvalid, F src_row, const float* gamma,
                                           float eps) {
  __shared__ float inv[GEMV_TP];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (gamma != nullptr && warp < GEMV_TP) {
    float ss = 0.f;
    if (warp < nvalid) {
      const float* x = src_row(warp);
      for (int k = lane; k < K; k += 32) ss = fmaf(x[k], x[k], ss);
    }
    ss = warp_sum(ss);
    if (lane == 0) inv[warp] = 1.0f / sqrtf(ss / (float)K + eps);
  }
  __syncthreads();
  for (int t = 0; t < GEMV_TP; ++t) {
    const float* x = t < nvalid ? src_row(t) : nullptr;
    const float sc = gamma != nullptr ? inv[t] : 1.f;
    for (int k = threadIdx.x; k < K; k += blockDim.x) {
      float v = 0.f;
      if (x) v = gamma != nullptr ? (x[k] * sc) * gamma[k] : x[k];
      xs[t * K + k] = v;
    }
  }
  __syncthreads();
}

// ---------------------------------------------------------------------------
// QKV projection + RoPE + paged KV write. A warp unit owns rows
// {i0, i0+1, i0+d/2, i0+1+d/2} of one head so both halves of each rotary
// pair are in the same warp. grid: (ceil(units/8), ceil(T/TP)).
template <class WT>
__global__ void __launch_bounds__(256) k_qkv(Dims D, DevState S, StepBuf B, const float* __restrict__ gamma,
                                             const WT* __restrict__ W, const float* __restrict__ scale,
                                             int layer, int T) {
  extern __shared__ __align__(16) float xs[];
  const int t0 = blockIdx.y * GEMV_TP;
  const int nvalid = min(GEMV_TP, T - t0);
  stage_rows(xs, D.h, nvalid, [&](int t) { return B.x + (size_t)(t0 + t) * D.h; }, gamma, D.eps);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q4 = D.d / 4;
  const int unit = blockIdx.x * GEMV_WARPS + warp;
  if (unit >= (D.Hq + 2 * D.Hkv) * q4) return;
  const int head = unit / q4, i0 = 2 * (unit % q4), half = D.d / 2;
  const int base = head * D.d;
  const int rows[4] = {base + i0, base + i0 + 1, base + i0 + half, base + i0 + 1 + half};
  const WT* wr[4];
#pragma unroll
  for (int r = 0; r < 4; ++r) wr[r] = W + (size_t)rows[r] * D.h;
  float acc[16];
  gemv_lane<WT, 4, GEMV_TP>(wr, D.h, xs, D.h, acc);
  const float val0 = reduce_scatter<16>(acc);
  const int v = (lane >> 1) & 15, r = v / GEMV_TP, t = v % GEMV_TP;
  const float val = scale != nullptr ? val0 * scale[rows[r]] : val0;
  const int pv = ((r ^ 2) * GEMV_TP + t) * 2;     // lane holding the rotary partner
  const float partner = __shfl_sync(0xffffffffu, val, pv);
  if ((lane & 1) || t >= nvalid) return;
  const int row = t0 + t;
  const int pos = B.row_pos[row];
  if (pos < 0 || pos >= D.max_ctx) { atomicOr(S.err, DERR_POS); return; }
  const int j = i0 + (r & 1);                      // rotary frequency index
  const int dim = (r < 2) ? j : j + half;
  float outv = val;
  if (head < D.Hq + D.Hkv) {
    const float c = S.rope_cos[(size_t)pos * half + j], s = S.rope_sin[(size_t)pos * half + j];
    // first half: a cos - b sin; second half: b cos + a sin (a = first-half value)
    outv = (r < 2) ? (val * c - partner * s) : (val * c + partner * s);
  }
  if (head < D.Hq) {
    B.q[((size_t)row * D.Hq + head) * D.d + dim] = outv;
    return;
  }
  const int is_v = head >= D.Hq + D.Hkv;
  const int hk = head - D.Hq - (is_v ? D.Hkv : 0);
  const int seq = B.row_seq[row];
  const int pi = pos / D.P;
  if (pi >= D.max_pages) { atomicOr(S.err, DERR_PAGE); return; }
  const int page = S.bt[(size_t)seq * D.max_pages + pi];
  if (page < 0) { atomicOr(S.err, DERR_PAGE); return; }
  const size_t off = (size_t)page * D.page_elems +
                     ((((size_t)layer * 2 + is_v) * D.Hkv + hk) * D.P + (pos % D.P)) * D.d + dim;
  if (D.act_f32) reinterpret_cast<float*>(S.kv)[off] = outv;
  else reinterpret_cast<uint16_t*>(S.kv)[off] = f_to_bf16(outv);
}

// ---------------------------------------------------------------------------
// Output projection + residual: x[t][o] += sum_k W_o[o][k] * attn[t][k].
template <class WT>
__global__ void __launch_bounds__(256) k_oproj(Dims D, StepBuf B, const WT* __restrict__ W,
                                               const float* __restrict__ scale, int T) {
  extern __shared__ __align__(16) float xs[];
  const int K = D.Hq * D.d;
  const int t0 = blockIdx.y * GEMV_TP;
  const int nvalid = min(GEMV_TP, T - t0);
  stage_rows(xs, K, nvalid, [&](int t) { return B.o + (size_t)(t0 + t) * K; }, nullptr, 0.f);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int unit = blockIdx.x * GEMV_WARPS + warp;
  if (unit * 4 >= D.h) return;
  const WT* wr[4];
#pragma unroll
  for (int r = 0; r < 4; ++r) wr[r] = W + (size_t)(unit * 4 + r) * K;
  float acc[16];
  gemv_lane<WT, 4, GEMV_TP>(wr, K, xs, K, acc);
  const float val = reduce_scatter<16>(acc);
  const int v = (lane >> 1) & 15, r = v / GEMV_TP, t = v % GEMV_TP;
  if ((lane & 1) || t >= nvalid) return;
  const int o = unit * 4 + r;
  const float y = scale != nullptr ? val * scale[o] : val;
  B.x[(size_t)(t0 + t) * D.h + o] += y;
}

// ---------------------------------------------------------------------------
// Expert gate/up + SwiGLU over the rows routed to one active expert.
// grid: (ceil(inter/4/8), active-expert slot, row pass). A warp unit owns 4
// gate rows and the same 4 up rows.
template <class WT>
__global__ void __launch_bounds__(256) k_gateup(Dims D, StepBuf B, const WT* __restrict__ Wg,
                                                const float* __restrict__ sg, const WT* __restrict__ Wu,
                                                const float* __restrict__ su) {
  extern __shared__ __align__(16) float xs[];
  const int slot = blockIdx.y;
  if (slot >= *B.n_active) return;
  const int cnt = B.act_cnt[slot], off = B.act_off[slot], e = B.act_expert[slot];
  const int p0 = blockIdx.z * GEMV_TP;
  if (p0 >= cnt) return;
  const int nvalid = min(GEMV_TP, cnt - p0);
  const int* pairs = B.perm + off + p0;
  stage_rows(xs, D.h, nvalid, [&](int t) { return B.u + (size_t)(pairs[t] / D.NS) * D.h; }, nullptr, 0.f);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int unit = blockIdx.x * GEMV_WARPS + warp;
  if (unit * 4 >= D.inter) return;
  const size_t ebase = (size_t)e * D.inter * D.h;
  const WT* wr[8];
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    wr[r] = Wg + ebase + (size_t)(unit * 4 + r) * D.h;
    wr[r + 4] = Wu + ebase + (size_t)(unit * 4 + r) * D.h;
  }
  float acc[32];
  gemv_lane<WT, 8, GEMV_TP>(wr, D.h, xs, D.h, acc);
  const float val = reduce_scatter<32>(acc);          // lane = r*TP + t
  const float up = __shfl_sync(0xffffffffu, val, (lane + 16) & 31);
  if (lane >= 16) return;
  const int r = lane / GEMV_TP, t = lane % GEMV_TP;
  if (t >= nvalid) return;
  const int j = unit * 4 + r;
  float g = val, uu = up;
  if (sg != nullptr) { g *= sg[(size_t)e * D.inter + j]; uu *= su[(size_t)e * D.inter + j]; }
  B.h_act[(size_t)pairs[t] * D.inter + j] = silu(g) * uu;
}

// Expert down projection y[pair][o] = sum_j W_d[e][o][j] * h_act[pair][j],
// then the combine: the last block to finish a 32-column tile of the output
// (over all expert slots and row passes) adds, for every row r and column o
// of the tile, sum over slots s (in order) of w[r][s] * y[r*NS + s][o] to the
// residual x (routed weight p, shared weight 1).
template <class WT>
__global__ void __launch_bounds__(256) k_down(Dims D, StepBuf B, const WT* __restrict__ Wd,
                                              const float* __restrict__ sd, int T) {
  extern __shared__ __align__(16) float xs[];
  __shared__ int s_last;
  const int slot = blockIdx.y;
  const int p0 = blockIdx.z * GEMV_TP;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int cnt = 0, off = 0, e = 0;
  bool work = slot < *B.n_active;
  if (work) {
    cnt = B.act_cnt[slot]; off = B.act_off[slot]; e = B.act_expert[slot];
    work = p0 < cnt;
  }
  if (work) {                                       // block-uniform branch
    const int nvalid = min(GEMV_TP, cnt - p0);
    const int* pairs = B.perm + off + p0;
    stage_rows(xs, D.inter, nvalid, [&](int t) { return B.h_act + (size_t)pairs[t] * D.inter; }, nullptr, 0.f);
    const int unit = blockIdx.x * GEMV_WARPS + warp;
    if (unit * 4 < D.h) {
      const WT* wr[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) wr[r] = Wd + ((size_t)e * D.h + unit * 4 + r) * D.inter;
      float acc[16];
      gemv_lane<WT, 4, GEMV_TP>(wr, D.inter, xs, D.inter, acc);
      const float val = reduce_scatter<16>(acc);
      const int v = (lane >> 1) & 15, r = v / GEMV_TP, t = v % GEMV_TP;
      if (!(lane & 1) && t < nvalid) {
        const int o = unit * 4 + r;
        B.y[(size_t)pairs[t] * D.h + o] = sd != nullptr ? val * sd[(size_t)e * D.h + o] : val;
      }
    }
  }
  __syncthreads();
  int* ctr = B.cnt_down + blockIdx.x;
  if (threadIdx.x == 0) {
    __threadfence();
    s_last = (atomicAdd(ctr, 1) == (int)(gridDim.y * gridDim.z) - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const int c0 = blockIdx.x * GEMV_WARPS * 4;
  const int ncol = min(GEMV_WARPS * 4, D.h - c0);
  for (int i = threadIdx.x; i < T * ncol; i += blockDim.x) {
    const int r = i / ncol, j = c0 + i % ncol;
    float acc = 0.f;
    for (int s2 = 0; s2 < D.NS; ++s2) {
      const float w = s2 < D.k ? B.wts[r * D.k + s2] : 1.f;
      acc = fmaf(w, __ldcg(B.y + ((size_t)r * D.NS + s2) * D.h + j), acc);
    }
    B.x[(size_t)r * D.h + j] += acc;
  }
  if (threadIdx.x == 0) *ctr = 0;
}

// ---------------------------------------------------------------------------
// Final RMSNorm + LM head + per-block argmax. Each block covers 32 vocab rows
// and writes one (max, index) candidate per activation row; ties keep the
// lowest index. grid: (ceil(V/32), ceil(T/TP)).
template <class WT>
__global__ void __launch_bounds__(256) k_lmhead(Dims D, StepBuf B, const WT* __restrict__ W,
                                                const float* __restrict__ gamma, const float* __restrict__ x,
                                                int T, float* __restrict__ logits_dbg, bool fused) {
  extern __shared__ __align__(16) float xs[];
  __shared__ float cand[GEMV_TP][GEMV_WARPS * 4];
  const int t0 = blockIdx.y * GEMV_TP;
  const int nvalid = min(GEMV_TP, T - t0);
  stage_rows(xs, D.h, nvalid, [&](int t) { return x + (size_t)(t0 + t) * D.h; }, gamma, D.eps);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row0 = (blockIdx.x * GEMV_WARPS + warp) * 4;
  float val = -INFINITY;
  int v = (lane >> 1) & 15, r = v / GEMV_TP, t = v % GEMV_TP;
  if (row0 < D.V) {   // V is a multiple of 4 (checked at init)
    const WT* wr[4];
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) wr[rr] = W + (size_t)(row0 + rr) * D.h;
    float acc[16];
    gemv_lane<WT, 4, GEMV_TP>(wr, D.h, xs, D.h, acc);
    val = reduce_scatter<16>(acc);
    if (logits_dbg != nullptr && !(lane & 1) && t < nvalid)
      logits_dbg[(size_t)(t0 + t) * D.V + row0 + r] = val;
  }
  if (!(lane & 1)) cand[t][warp * 4 + r] = val;
  __syncthreads();
  if (threadIdx.x < nvalid) {
    const int tt = threadIdx.x;
    float best = -INFINITY;
    int bi = -1;
    for (int i = 0; i < GEMV_WARPS * 4; ++i) {
      const int vi = blockIdx.x * GEMV_WARPS * 4 + i;
      if (vi >= D.V) break;
      const float c = cand[tt][i];
      if (bi < 0 || c > best) { best = c; bi = vi; }
    }
    B.am_val[(size_t)(t0 + tt) * B.n_vblocks + blockIdx.x] = best;
    B.am_idx[(size_t)(t0 + tt) * B.n_vblocks + blockIdx.x] = bi;
  }
  if (!fused) return;
  // the last block of this row pass reduces every block's candidate:
  // larger value wins, equal values keep the lower index
  __shared__ int s_last;
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    s_last = (atomicAdd(B.cnt_lm + blockIdx.y, 1) == (int)gridDim.x - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  if (warp < nvalid) {
    const size_t base = (size_t)(t0 + warp) * B.n_vblocks;
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    for (int i = lane; i < B.n_vblocks; i += 32) {
      const float c = __ldcg(B.am_val + base + i);
      const int ci = __ldcg(B.am_idx + base + i);
      if (c > bv || (c == bv && ci < bi)) { bv = c; bi = ci; }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
    }
    if (lane == 0) B.g[t0 + warp] = bi;
  }
  if (threadIdx.x == 0) B.cnt_lm[blockIdx.y] = 0;
}

// Reduce the per-block candidates of each row: larger value wins, equal
// values keep the lower vocabulary index (a total order, so the tree shape
// cannot change the result).
__global__ void k_argmax_reduce(StepBuf B, int T, int* out) {
  const int r = blockIdx.x;
  __shared__ float sv[256];
  __shared__ int si[256];
  float best = -INFINITY;
  int bi = 0x7fffffff;
  for (int i = threadIdx.x; i < B.n_vblocks; i += blockDim.x) {
    const float c = B.am_val[(size_t)r * B.n_vblocks + i];
    const int ci = B.am_idx[(size_t)r * B.n_vblocks + i];
    if (c > best || (c == best && ci < bi)) { best = c; bi = ci; }
  }
  sv[threadIdx.x] = best;
  si[threadIdx.x] = bi;
  __syncthreads();
  for (int s = blockDim.x / 2; s > 0; s >>= 1) {
    if (threadIdx.x < s) {
      const float c = sv[threadIdx.x + s];
      const int ci = si[threadIdx.x + s];
      if (c > sv[threadIdx.x] || (c == sv[threadIdx.x] && ci < si[threadIdx.x])) {
        sv[threadIdx.x] = c;
        si[threadIdx.x] = ci;
      }
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) out[r] = si[0];
}

// ---------------------------------------------------------------------------
// launchers
static inline int cdiv(int a, int b) { return (a + b - 1) / b; }


cudaError_t configure_gemv_kernels() {
  cudaError_t e = cudaSuccess, r;
#define ALLOW(k) if ((r = allow_dyn_smem(k)) != cudaSuccess) e = r
  ALLOW(k_qkv<float>); ALLOW(k_qkv<bf16_t>); ALLOW(k_qkv<fp8_t>);
  ALLOW(k_oproj<float>); ALLOW(k_oproj<bf16_t>); ALLOW(k_oproj<fp8_t>);
  ALLOW(k_gateup<float>); ALLOW(k_gateup<bf16_t>); ALLOW(k_gateup<fp8_t>);
  ALLOW(k_down<float>); ALLOW(k_down<bf16_t>); ALLOW(k_down<fp8_t>);
  ALLOW(k_lmhead<float>); ALLOW(k_lmhead<bf16_t>);
#undef ALLOW
  return e;
}

void launch_qkv(const Dims& D, const DevState& S, const StepBuf& B, const LayerW& W, int layer, int T,
                cudaStream_t st) {
  const int units = (D.Hq + 2 * D.Hkv) * (D.d / 4);
  dim3 grid(cdiv(units, GEMV_WARPS), cdiv(T, GEMV_TP));
  const size_t sm = (size_t)GEMV_TP * D.h * sizeof(float);
  switch (D.wdtype) {
    case 0: k_qkv<float><<<grid, 256, sm, st>>>(D, S, B, W.attn_norm, (const float*)W.w_qkv, nullptr, layer, T); break;
    case 1: k_qkv<bf16_t><<<grid, 256, sm, st>>>(D, S, B, W.attn_norm, (const bf16_t*)W.w_qkv, nullptr, layer, T); break;
    default: k_qkv<fp8_t><<<grid, 256, sm, st>>>(D, S, B, W.attn_norm, (const fp8_t*)W.w_qkv, W.s_qkv, layer, T);
  }
}

void launch_oproj(const Dims& D, const StepBuf& B, const LayerW& W, int T, cudaStream_t st) {
  dim3 grid(cdiv(D.h / 4, GEMV_WARPS), cdiv(T, GEMV_TP));
  const size_t sm = (size_t)GEMV_TP * D.Hq * D.d * sizeof(float);
  switch (D.wdtype) {
    case 0: k_oproj<float><<<grid, 256, sm, st>>>(D, B, (const float*)W.w_o, nullptr, T); break;
    case 1: k_oproj<bf16_t><<<grid, 256, sm, st>>>(D, B, (const bf16_t*)W.w_o, nullptr, T); break;
    default: k_oproj<fp8_t><<<grid, 256, sm, st>>>(D, B, (const fp8_t*)W.w_o, W.s_o, T);
  }
}

void launch_gateup(const Dims& D, const StepBuf& B, const LayerW& W, int T, cudaStream_t st) {
  const int max_active = (D.E > 0 ? (D.E < T * D.k ? D.E : T * D.k) : 0) + D.S;
  dim3 g1(cdiv(D.inter / 4, GEMV_WARPS), max_active, cdiv(T, GEMV_TP));
  const size_t sm1 = (size_t)GEMV_TP * D.h * sizeof(float);
  switch (D.wdtype) {
    case 0: k_gateup<float><<<g1, 256, sm1, st>>>(D, B, (const float*)W.w_gate, nullptr, (const float*)W.w_up, nullptr); break;
    case 1: k_gateup<bf16_t><<<g1, 256, sm1, st>>>(D, B, (const bf16_t*)W.w_gate, nullptr, (const bf16_t*)W.w_up, nullptr); break;
    default: k_gateup<fp8_t><<<g1, 256, sm1, st>>>(D, B, (const fp8_t*)W.w_gate, W.s_gate, (const fp8_t*)W.w_up, W.s_up);
  }
}

void launch_down(const Dims& D, const StepBuf& B, const LayerW& W, int T, cudaStream_t st) {
  const int max_active = (D.E > 0 ? (D.E < T * D.k ? D.E : T * D.k) : 0) + D.S;
  dim3 g2(cdiv(D.h / 4, GEMV_WARPS), max_active, cdiv(T, GEMV_TP));
  const size_t sm2 = (size_t)GEMV_TP * D.inter * sizeof(float);
  switch (D.wdtype) {
    case 0: k_down<float><<<g2, 256, sm2, st>>>(D, B, (const float*)W.w_down, nullptr, T); break;
    case 1: k_down<bf16_t><<<g2, 256, sm2, st>>>(D, B, (const bf16_t*)W.w_down, nullptr, T); break;
    default: k_down<fp8_t><<<g2, 256, sm2, st>>>(D, B, (const fp8_t*)W.w_down, W.s_down, T);
  }
}

void launch_lmhead(const Dims& D, const StepBuf& B, const void* lm_head, const float* final_norm,
                   const float* x, int T, float* logits_dbg, bool fuse_argmax, cudaStream_t st) {
  dim3 grid(B.n_vblocks, cdiv(T, GEMV_TP));
  const size_t sm = (size_t)GEMV_TP * D.h * sizeof(float);
  if (D.act_f32) {
    k_lmhead<float><<<grid, 256, sm, st>>>(D, B, (const float*)lm_head, final_norm, x, T, logits_dbg,
                                           fuse_argmax);
  } else {
    k_lmhead<bf16_t><<<grid, 256, sm, st>>>(D, B, (const bf16_t*)lm_head, final_norm, x, T, logits_dbg,
                                            fuse_argmax);
  }
}

void launch_argmax(const StepBuf& B, int T, cudaStream_t st) { k_argmax_reduce<<<T, 256, 0, st>>>(B, T, B.g); }

}  // namespace spec
