// Shared building blocks of the weight-streaming GEMV kernels.
//
// A warp owns R weight rows ("a unit") and streams them with 16-byte
// non-allocating loads, 32 lanes side by side; each lane accumulates its
// chunks in increasing order and a fixed butterfly reduce-scatter combines
// the lanes. Nothing in an output's arithmetic depends on T, on the row's
// place in the batch or on the launch shape.
#pragma once
#include "common.cuh"

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
// Streaming variant: activation rows are read from global memory (through L1)
// instead of shared memory, optionally scaled by gamma per column; the first
// group of a unit's weight chunks can be loaded ahead (before the kernel waits
// for its predecessor, or before the previous unit's reduction).
template <class WT, int R, int G>
__device__ __forceinline__ void load_group(uint4 (&wv)[G][R], const WT* const (&wr)[R], int nch, int c0) {
  constexpr int EP = Elt<WT>::per16;
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const int c = c0 + 32 * g;
#pragma unroll
    for (int r = 0; r < R; ++r) wv[g][r] = c < nch ? ld_stream(wr[r] + (size_t)c * EP) : make_uint4(0, 0, 0, 0);
  }
}

template <class WT, int R, int TP, int Q>
__device__ __forceinline__ void fma_q(const uint4 (&wv)[R], const float* const (&xr)[TP], const float* gamma, int k,
                                      float (&acc)[R * TP]) {
  float4 gq = make_float4(1.f, 1.f, 1.f, 1.f);
  if (gamma != nullptr) gq = __ldg(reinterpret_cast<const float4*>(gamma + k + 4 * Q));
  float xv[TP][4];
#pragma unroll
  for (int t = 0; t < TP; ++t) {
    float4 x4 = make_float4(0.f, 0.f, 0.f, 0.f);
    if (xr[t] != nullptr) x4 = __ldg(reinterpret_cast<const float4*>(xr[t] + k + 4 * Q));
    xv[t][0] = x4.x * gq.x; xv[t][1] = x4.y * gq.y; xv[t][2] = x4.z * gq.z; xv[t][3] = x4.w * gq.w;
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

// acc[r*TP + t] = sum_k W[row r][k] * (gamma[k]) * x_t[k] over this lane's
// chunks in increasing order. wv holds the unit's first chunk group on entry.
template <class WT, int R, int TP, int G>
__device__ __forceinline__ void unit_dot(uint4 (&wv)[G][R], const WT* const (&wr)[R], int K,
                                         const float* const (&xr)[TP], const float* gamma, float (&acc)[R * TP]) {
  constexpr int EP = Elt<WT>::per16;
  const int nch = K / EP, lane = threadIdx.x & 31;
#pragma unroll
  for (int i = 0; i < R * TP; ++i) acc[i] = 0.f;
  for (int c0 = lane; c0 < nch; c0 += 32 * G) {
    if (c0 != lane) load_group<WT, R, G>(wv, wr, nch, c0);
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const int c = c0 + 32 * g;
      if (c < nch) {
        const int k = c * EP;
        fma_q<WT, R, TP, 0>(wv[g], xr, gamma, k, acc);
        if constexpr (EP >= 8) fma_q<WT, R, TP, 1>(wv[g], xr, gamma, k, acc);
        if constexpr (EP >= 16) {
          fma_q<WT, R, TP, 2>(wv[g], xr, gamma, k, acc);
          fma_q<WT, R, TP, 3>(wv[g], xr, gamma, k, acc);
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Paired accumulation: each output keeps two partial sums -- even and odd
// elements of every chunk, in increasing chunk order -- updated by one packed
// fma.rn.f32x2 (each half rounds exactly like fmaf), and returns their sum.
__device__ __forceinline__ unsigned long long pack2(float a, float b) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ float sum2(unsigned long long v) {
  float a, b;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
  return a + b;
}
__device__ __forceinline__ void ffma2(unsigned long long& acc, unsigned long long w, unsigned long long x) {
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(w), "l"(x));
}

// Four elements of group Q of a 16-byte weight vector as two packed pairs.
template <class WT, int Q>
__device__ __forceinline__ void wpairs(const uint4& v, unsigned long long& p0, unsigned long long& p1) {
  float w[4];
  unpack4<WT, Q>(v, w);
  p0 = pack2(w[0], w[1]);
  p1 = pack2(w[2], w[3]);
}

template <class WT, int R, int TP, int Q>
__device__ __forceinline__ void fma2_q(const uint4 (&wv)[R], const float* const (&xr)[TP], int k,
                                       unsigned long long (&acc)[R * TP]) {
  unsigned long long xa[TP], xb[TP];
#pragma unroll
  for (int t = 0; t < TP; ++t) {
    float4 x4 = make_float4(0.f, 0.f, 0.f, 0.f);
    if (xr[t] != nullptr) x4 = *reinterpret_cast<const float4*>(xr[t] + k + 4 * Q);
    xa[t] = pack2(x4.x, x4.y);
    xb[t] = pack2(x4.z, x4.w);
  }
#pragma unroll
  for (int r = 0; r < R; ++r) {
    unsigned long long w0, w1;
    wpairs<WT, Q>(wv[r], w0, w1);
#pragma unroll
    for (int t = 0; t < TP; ++t) {
      ffma2(acc[r * TP + t], w0, xa[t]);
      ffma2(acc[r * TP + t], w1, xb[t]);
    }
  }
}

// out[r*TP + t] = sum_k W[row r][k] * x_t[k] over this lane's chunks
// (increasing order, even/odd pairs). x rows may live in shared or global
// memory (plain loads); wv holds the unit's first chunk group on entry.
template <class WT, int R, int TP, int G>
__device__ __forceinline__ void unit_dot2(uint4 (&wv)[G][R], const WT* const (&wr)[R], int K,
                                          const float* const (&xr)[TP], float (&out)[R * TP]) {
  constexpr int EP = Elt<WT>::per16;
  const int nch = K / EP, lane = threadIdx.x & 31;
  unsigned long long acc[R * TP];
#pragma unroll
  for (int i = 0; i < R * TP; ++i) acc[i] = 0ull;
  for (int c0 = lane; c0 < nch; c0 += 32 * G) {
    if (c0 != lane) load_group<WT, R, G>(wv, wr, nch, c0);
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const int c = c0 + 32 * g;
      if (c < nch) {
        const int k = c * EP;
        fma2_q<WT, R, TP, 0>(wv[g], xr, k, acc);
        if constexpr (EP >= 8) fma2_q<WT, R, TP, 1>(wv[g], xr, k, acc);
        if constexpr (EP >= 16) {
          fma2_q<WT, R, TP, 2>(wv[g], xr, k, acc);
          fma2_q<WT, R, TP, 3>(wv[g], xr, k, acc);
        }
      }
    }
  }
#pragma unroll
  for (int i = 0; i < R * TP; ++i) out[i] = sum2(acc[i]);
}

// Stage rows [t0, t0 + n) of x (row stride K) into xs[TP][K] as
// (x * inv[t]) * gamma[k] (gamma may be null: plain copy); zeros past n.
__device__ __forceinline__ void stage_norm(float* xs, const float* x, int t0, int n, int K, const float* inv,
                                           const float* gamma) {
  const int K4 = K / 4;
#pragma unroll 4
  for (int i = threadIdx.x; i < GEMV_TP * K4; i += blockDim.x) {
    const int t = i / K4, k4 = i % K4;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (t < n) {
      v = reinterpret_cast<const float4*>(x + (size_t)(t0 + t) * K)[k4];
      if (gamma != nullptr) {
        const float s = inv[t0 + t];
        const float4 g = reinterpret_cast<const float4*>(gamma)[k4];
        v = make_float4((v.x * s) * g.x, (v.y * s) * g.y, (v.z * s) * g.z, (v.w * s) * g.w);
      }
    }
    reinterpret_cast<float4*>(xs)[i] = v;
  }
}

// One element of the expert combine: x[t][kcol] + sum over slots s (in
// order) of w[t][s] * y[t*NS + s][kcol] (routed weight p, shared weight 1).
__device__ __forceinline__ float combine_one(const float* x, const float* y, const float* wts, int t, int kcol,
                                             int K, int NS, int k) {
  float a = 0.f;
  for (int s = 0; s < NS; ++s) {
    const float w = s < k ? wts[t * k + s] : 1.f;
    a = fmaf(w, y[((size_t)t * NS + s) * K + kcol], a);
  }
  return x[(size_t)t * K + kcol] + a;
}

// Inverse RMS of rows [0, T) of x into inv[] (shared), warp r handling rows
// r, r+8, ...: 1 / sqrt(mean(x^2) + eps). Each lane issues up to eight
// float4 loads at once (K must be a multiple of 4); lane partials are added in
// a fixed order, so the result depends only on the row.
__device__ __forceinline__ void row_inv_rms(const float* x, int T, int K, float eps, float* inv) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int K4 = K / 4;
  for (int r = warp; r < T; r += blockDim.x / 32) {
    const float4* xr = reinterpret_cast<const float4*>(x + (size_t)r * K);
    float ss = 0.f;
    for (int b = lane; b < K4; b += 32 * 8) {
      float4 v[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = (b + 32 * i < K4) ? xr[b + 32 * i] : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        ss = fmaf(v[i].x, v[i].x, ss); ss = fmaf(v[i].y, v[i].y, ss);
        ss = fmaf(v[i].z, v[i].z, ss); ss = fmaf(v[i].w, v[i].w, ss);
      }
    }
    ss = warp_sum(ss);
    if (lane == 0) inv[r] = 1.0f / sqrtf(ss / (float)K + eps);
  }
}

// ---------------------------------------------------------------------------
// Warp tensor-core GEMV (bf16 / e4m3 weights, at most 8 activation columns):
// mma.sync m16n8k16 with A = 16 weight rows, B = 8 columns (tokens or routed
// pairs), C = fp32. Lane (g, q) = (lane / 4, lane % 4) streams 16 contiguous
// bytes of weight rows g and g + 8 per step -- 8 bf16 (or 16 e4m3 widened to
// bf16) at k = kb + EPL * q -- and those bytes are the lane's A fragment as
// they are: the MMA's K slots are a permutation of the step's k values, and
// the B fragment (column g's activations at the same k) uses the same one.
// For MMA j of a 8-element group starting at k0: A slots (2q, 2q+1) <- k0 +
// 4j + {0,1}, slots (2q+8, 2q+9) <- k0 + 4j + {2,3}. Activations are fp32,
// split into bf16 hi + lo (two MMAs, two accumulators added at the end), so
// a column's result keeps near-fp32 precision and depends only on that
// column's own inputs. Result: c[0], c[1] = rows g x columns 2q, 2q+1;
// c[2], c[3] = rows g + 8 x the same columns.
__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// x, y -> bf16x2 hi = (bf16(x), bf16(y)) and lo = (bf16(x - hi.x), bf16(y - hi.y)),
// x in the low half (the lower k index).
__device__ __forceinline__ void split_bf16x2(float x, float y, uint32_t& hi, uint32_t& lo) {
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(hi) : "f"(y), "f"(x));
  const float xh = __uint_as_float(hi << 16), yh = __uint_as_float(hi & 0xFFFF0000u);
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(lo) : "f"(y - yh), "f"(x - xh));
}

// Eight e4m3 values (two 32-bit words) -> four bf16x2 words, exactly.
__device__ __forceinline__ void e4m3x8_bf16(uint32_t w0, uint32_t w1, uint32_t (&o)[4]) {
  const uint32_t w[2] = {w0, w1};
#pragma unroll
  for (int i = 0; i < 2; ++i) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)((w[i] >> (16 * h)) & 0xFFFF), __NV_E4M3);
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hr));
      o[2 * i + h] = (__float_as_uint(f.x) >> 16) | (__float_as_uint(f.y) & 0xFFFF0000u);
    }
  }
}

template <class WT> struct MmaStep;                   // k values one step covers (4 lanes x EPL)
template <> struct MmaStep<bf16_t> { static constexpr int EPL = 8, K = 32; };
template <> struct MmaStep<fp8_t> { static constexpr int EPL = 16, K = 64; };
template <> struct MmaStep<fp4_t> { static constexpr int EPL = 32, K = 128; };

template <class WT> struct IsQ4 { static constexpr bool v = false; };
template <> struct IsQ4<fp4_t> { static constexpr bool v = true; };

// Element k of a weight row (an nvfp4 row holds two elements per byte).
template <class WT>
__device__ __forceinline__ const WT* at_k(const WT* row, int k) {
  if constexpr (IsQ4<WT>::v) return row + (k >> 1);
  else return row + k;
}

// Row r of matrix e in a stack of [rows][K] matrices. An nvfp4 stack holds
// one record per matrix -- the codes of all rows (K / 2 bytes a row), then
// the block-scale codes (K / 16 a row) -- and *sc gets the row's scales.
template <class WT>
__device__ __forceinline__ const WT* stack_row(const WT* W, int e, int rows, int r, int K, const uint8_t** sc) {
  if constexpr (IsQ4<WT>::v) {
    const uint8_t* rec = reinterpret_cast<const uint8_t*>(W) + (size_t)e * rows * (K / 2 + K / 16);
    *sc = rec + (size_t)rows * (K / 2) + (size_t)r * (K / 16);
    return reinterpret_cast<const WT*>(rec + (size_t)r * (K / 2));
  } else {
    *sc = nullptr;
    return W + ((size_t)e * rows + r) * K;
  }
}

// nvfp4 block scales of a unit's two rows: the row pointers and, per loaded
// step, the lane's two scale codes (its 32 elements span two 16-element blocks).
template <int NB> struct Q4Scales {
  const uint8_t* lo = nullptr;
  const uint8_t* hi = nullptr;
  uint32_t a[NB], b[NB];
};

// Eight E2M1 codes (one word, element i in nibble i) times the E4M3 block
// scale `sc` -> four f16x2 words (element 2j in the low half of word j).
// Every product is exact in f16: at most 2 x 4 significant bits, magnitudes
// 2^-10 .. 2688.
__device__ __forceinline__ void q4x8_f16(uint32_t w, uint32_t sc, uint32_t (&o)[4]) {
  const __half_raw sr = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)(sc & 0xFF), __NV_E4M3);
  const __half2 s2 = __halves2half2(__half(sr), __half(sr));
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const __half2_raw hr = __nv_cvt_fp4x2_to_halfraw2((__nv_fp4x2_storage_t)((w >> (8 * j)) & 0xFF), __NV_E2M1);
    const __half2 v = __hmul2(__half2(hr), s2);
    o[j] = *reinterpret_cast<const uint32_t*>(&v);
  }
}

__device__ __forceinline__ void mma16816_f16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                             uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// mma_group8 with f16 weights: the activations enter as NP f16 parts of
// x * F16_OP_SCALE (each part the rounding of what the earlier ones leave).
template <int NP>
__device__ __forceinline__ void mma_group8_f16(float (&c)[NP][4], const uint32_t (&wa)[4], const uint32_t (&wb)[4],
                                               const float4& x0, const float4& x1) {
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const float4 v = half ? x1 : x0;
    float r[4] = {v.x * F16_OP_SCALE, v.y * F16_OP_SCALE, v.z * F16_OP_SCALE, v.w * F16_OP_SCALE};
#pragma unroll
    for (int part = 0; part < NP; ++part) {
      uint32_t b0, b1;
      asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(b0) : "f"(r[1]), "f"(r[0]));
      asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(b1) : "f"(r[3]), "f"(r[2]));
      mma16816_f16(c[part], wa[2 * half], wb[2 * half], wa[2 * half + 1], wb[2 * half + 1], b0, b1);
      if (part + 1 < NP) {
        r[0] -= f16_to_f((uint16_t)(b0 & 0xFFFF));
        r[1] -= f16_to_f((uint16_t)(b0 >> 16));
        r[2] -= f16_to_f((uint16_t)(b1 & 0xFFFF));
        r[3] -= f16_to_f((uint16_t)(b1 >> 16));
      }
    }
  }
}

// NP MMAs (activation parts) of one 8-element group: weights wa (row g) / wb
// (row g+8) as four bf16x2 words, activations x[0..8) of column g at the
// group's k. NP = 2: hi = bf16(x), lo = bf16(x - hi) (~16 bits); NP = 3 adds
// lo2 = bf16(x - hi - lo) (the full fp32 significand), for the projection
// whose outputs are rounded to bf16 for storage (the K/V cache), where a
// value's rounding must not depend on the split.
template <int NP>
__device__ __forceinline__ void mma_group8(float (&c)[NP][4], const uint32_t (&wa)[4], const uint32_t (&wb)[4],
                                           const float4& x0, const float4& x1) {
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const float4 v = half ? x1 : x0;
    float r[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int part = 0; part < NP; ++part) {
      uint32_t b0, b1;
      asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(b0) : "f"(r[1]), "f"(r[0]));
      asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(b1) : "f"(r[3]), "f"(r[2]));
      mma16816(c[part], wa[2 * half], wb[2 * half], wa[2 * half + 1], wb[2 * half + 1], b0, b1);
      if (part + 1 < NP) {
        r[0] -= __uint_as_float(b0 << 16);
        r[1] -= __uint_as_float(b0 & 0xFFFF0000u);
        r[2] -= __uint_as_float(b1 << 16);
        r[3] -= __uint_as_float(b1 & 0xFFFF0000u);
      }
    }
  }
}

// Block-split units: the 8 warps of a block share one 16-row unit and split
// its K steps -- warp w takes steps w, w + 8, w + 16, ... -- in batches of NB
// steps whose loads are all in flight at once; block_sum4 then adds the
// warps' partial c[4] in warp order (a fixed order) for warp 0.
template <class WT, int NB>
__device__ __forceinline__ void mma_load_batch(uint4 (&va)[NB], uint4 (&vb)[NB], const WT* wlo, const WT* whi,
                                               int K, int s0, Q4Scales<NB>& qs) {
  constexpr int SK = MmaStep<WT>::K, EPL = MmaStep<WT>::EPL;
  const int q = threadIdx.x & 3, nsteps = K / SK;
#pragma unroll
  for (int u = 0; u < NB; ++u) {
    const int st = s0 + 8 * u;
    const int k = st * SK + EPL * q;
    va[u] = st < nsteps ? ld_stream(at_k(wlo, k)) : make_uint4(0, 0, 0, 0);
    vb[u] = st < nsteps ? ld_stream(at_k(whi, k)) : make_uint4(0, 0, 0, 0);
    if constexpr (IsQ4<WT>::v) {   // the two block scales of the lane's 32 elements (k / 16 is even)
      qs.a[u] = st < nsteps ? (uint32_t)__ldg(reinterpret_cast<const unsigned short*>(qs.lo + k / 16)) : 0u;
      qs.b[u] = st < nsteps ? (uint32_t)__ldg(reinterpret_cast<const unsigned short*>(qs.hi + k / 16)) : 0u;
    }
  }
}

// This warp's partial c[4] of the unit (weight rows g / g + 8 against column
// x, nullptr = zeros). va/vb hold the warp's first batch on entry
// (mma_load_batch at s0 = warp).
// One K step of a unit for this lane: its 16-byte pieces of rows g (va) and
// g + 8 (vb) at k = step * SK + EPL * q, (nvfp4) their block-scale code pairs
// sa / sb, against column x (nullptr = zeros), into the NP part accumulators.
template <class WT, int NP>
__device__ __forceinline__ void mma_step(const uint4& va, const uint4& vb, uint32_t sa, uint32_t sb, int k,
                                         const float* x, float (&cp)[NP][4]) {
  constexpr int EPL = MmaStep<WT>::EPL;
#pragma unroll
  for (int h = 0; h < EPL / 8; ++h) {
    uint32_t wa[4], wb[4];
    float4 x0 = make_float4(0.f, 0.f, 0.f, 0.f), x1 = x0;
    if (x != nullptr) {
      x0 = *reinterpret_cast<const float4*>(x + k + 8 * h);
      x1 = *reinterpret_cast<const float4*>(x + k + 8 * h + 4);
    }
    if constexpr (IsQ4<WT>::v) {
      // group h: elements k + 8h .. k + 8h + 7, block scale h / 2 of the lane's pair
      const uint32_t ca = h == 0 ? va.x : h == 1 ? va.y : h == 2 ? va.z : va.w;
      const uint32_t cb = h == 0 ? vb.x : h == 1 ? vb.y : h == 2 ? vb.z : vb.w;
      q4x8_f16(ca, sa >> (8 * (h >> 1)), wa);
      q4x8_f16(cb, sb >> (8 * (h >> 1)), wb);
      mma_group8_f16<NP>(cp, wa, wb, x0, x1);
    } else {
      if constexpr (EPL == 8) {
        wa[0] = va.x; wa[1] = va.y; wa[2] = va.z; wa[3] = va.w;
        wb[0] = vb.x; wb[1] = vb.y; wb[2] = vb.z; wb[3] = vb.w;
      } else {
        e4m3x8_bf16(h ? va.z : va.x, h ? va.w : va.y, wa);
        e4m3x8_bf16(h ? vb.z : vb.x, h ? vb.w : vb.y, wb);
      }
      mma_group8<NP>(cp, wa, wb, x0, x1);
    }
  }
}

// The unit's result for this lane: the parts' accumulators added in part order.
template <int NP>
__device__ __forceinline__ void sum_parts(const float (&cp)[NP][4], float (&c)[4]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float t = cp[0][i];
#pragma unroll
    for (int part = 1; part < NP; ++part) t += cp[part][i];
    c[i] = t;
  }
}

template <class WT, int NB, int NP = 2>
__device__ __forceinline__ void mma_part(uint4 (&va)[NB], uint4 (&vb)[NB], const WT* wlo, const WT* whi, int K,
                                         const float* x, float (&c)[4], Q4Scales<NB>& qs) {
  constexpr int SK = MmaStep<WT>::K, EPL = MmaStep<WT>::EPL;
  const int q = threadIdx.x & 3, w = threadIdx.x >> 5, nsteps = K / SK;
  float cp[NP][4];
#pragma unroll
  for (int part = 0; part < NP; ++part)
#pragma unroll
    for (int i = 0; i < 4; ++i) cp[part][i] = 0.f;
  for (int s0 = w; s0 < nsteps; s0 += 8 * NB) {
    if (s0 != w) mma_load_batch<WT, NB>(va, vb, wlo, whi, K, s0, qs);
#pragma unroll
    for (int u = 0; u < NB; ++u) {
      const int st = s0 + 8 * u;
      if (st < nsteps) {
        uint32_t sa = 0, sb = 0;
        if constexpr (IsQ4<WT>::v) { sa = qs.a[u]; sb = qs.b[u]; }
        mma_step<WT, NP>(va[u], vb[u], sa, sb, st * SK + EPL * q, x, cp);
      }
    }
  }
  sum_parts<NP>(cp, c);
}

// Sum of the 8 warps' c[4] in warp order into warp 0's c (one barrier). red:
// shared [2][8][32] float4, alternated by the caller's unit parity, so the
// next unit's writes never meet warp 0's reads of this one.
__device__ __forceinline__ void block_sum4(float (&c)[4], float4* red, int parity) {
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float4* r = red + parity * 256;
  r[w * 32 + lane] = make_float4(c[0], c[1], c[2], c[3]);
  __syncthreads();
  if (w == 0) {
    float4 t = r[lane];
#pragma unroll
    for (int i = 1; i < 8; ++i) {
      const float4 v = r[i * 32 + lane];
      t.x += v.x; t.y += v.y; t.z += v.z; t.w += v.w;
    }
    c[0] = t.x; c[1] = t.y; c[2] = t.z; c[3] = t.w;
  }
}

// block_sum4 for the 8 warps 0..7 of a block that has more warps: the same
// order and buffers, with named barrier 1 (256 threads) for the block barrier.
__device__ __forceinline__ void block_sum4_w8(float (&c)[4], float4* red, int parity) {
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float4* r = red + parity * 256;
  r[w * 32 + lane] = make_float4(c[0], c[1], c[2], c[3]);
  asm volatile("bar.sync 1, 256;" ::: "memory");
  if (w == 0) {
    float4 t = r[lane];
#pragma unroll
    for (int i = 1; i < 8; ++i) {
      const float4 v = r[i * 32 + lane];
      t.x += v.x; t.y += v.y; t.z += v.z; t.w += v.w;
    }
    c[0] = t.x; c[1] = t.y; c[2] = t.z; c[3] = t.w;
  }
}

}  // namespace spec
