// Device helpers shared by the verify-step kernels (sm_103a).
#pragma once
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_fp4.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "kernels.h"

namespace spec {

constexpr int WARP = 32;

// Error bits a kernel may raise (read back by the host after a step).
enum : int { DERR_PAGE = 1, DERR_TOKEN = 2, DERR_POS = 4, DERR_TIMEOUT = 8 };

// Longest time one wait on an mbarrier may take before the kernel gives up
// (sets DERR_TIMEOUT, stops issuing work, frees what it holds and returns).
constexpr unsigned long long WAIT_DEADLINE_NS = 250ull * 1000 * 1000;

__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait for phase `parity` of the mbarrier at shared address `bar`. Returns
// false once WAIT_DEADLINE_NS have passed, or as soon as another thread of
// the grid has raised DERR_TIMEOUT in *err (then every waiter gives up
// together instead of each spending its own deadline).
__device__ __forceinline__ bool mbar_wait_deadline(uint32_t bar, uint32_t parity, const int* err) {
  auto try_once = [&]() {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0;
  };
  for (int i = 0; i < 32; ++i)
    if (try_once()) return true;
  const unsigned long long t0 = globaltimer_ns();
  for (;;) {
    if (try_once()) return true;
    if (globaltimer_ns() - t0 > WAIT_DEADLINE_NS) return false;
    if (err != nullptr && (*reinterpret_cast<const volatile int*>(err) & DERR_TIMEOUT)) return false;
  }
}

// ---- storage element types --------------------------------------------------
struct bf16_t { uint16_t v; };
struct fp8_t { uint8_t v; };
struct fp4_t { uint8_t v; };     // two E2M1 codes: element 2j in the low nibble of byte j

template <class T> struct Elt;
template <> struct Elt<float>  { static constexpr int per16 = 4; };
template <> struct Elt<bf16_t> { static constexpr int per16 = 8; };
template <> struct Elt<fp8_t>  { static constexpr int per16 = 16; };

__device__ __forceinline__ float bf16_to_f(uint16_t b) { return __uint_as_float(((uint32_t)b) << 16); }

__device__ __forceinline__ uint16_t f_to_bf16(float f) {
  __nv_bfloat16 h = __float2bfloat16_rn(f);
  return *reinterpret_cast<uint16_t*>(&h);
}

// Operand parts of the tensor-core GEMMs. bf16 models: parts of x in bf16.
// e4m3-weight models: parts of x * F16_OP_SCALE in f16 (the MMA runs on f16,
// to which e4m3 widens in one instruction; f16 hi + lo keeps ~22 bits, and
// the exact power-of-two scale keeps the lo parts of the activations, which
// stay far below 255 in magnitude, clear of f16's subnormal range). The
// GEMM epilogue multiplies by 1 / F16_OP_SCALE.
constexpr float F16_OP_SCALE = 256.0f;
__device__ __forceinline__ uint16_t f_to_f16(float f) { return __half_as_ushort(__float2half_rn(f)); }
__device__ __forceinline__ float f16_to_f(uint16_t b) { return __half2float(__ushort_as_half(b)); }
// Split x into n_parts 16-bit parts (bf16 or, with f16, of x * F16_OP_SCALE),
// each the rounding of what the earlier parts leave.
__device__ __forceinline__ void split_parts(float x, int f16, int n_parts, uint16_t* out) {
  float r = f16 ? x * F16_OP_SCALE : x;
  for (int i = 0; i < n_parts; ++i) {
    const uint16_t p = f16 ? f_to_f16(r) : f_to_bf16(r);
    out[i] = p;
    r -= f16 ? f16_to_f(p) : bf16_to_f(p);
  }
}

// 16-byte streaming load that does not allocate in L1 (weights are read once).
__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}

// Unpack one 16-byte vector into per16 floats.
template <class T> __device__ __forceinline__ void unpack(const uint4& v, float* o);

template <> __device__ __forceinline__ void unpack<float>(const uint4& v, float* o) {
  o[0] = __uint_as_float(v.x); o[1] = __uint_as_float(v.y);
  o[2] = __uint_as_float(v.z); o[3] = __uint_as_float(v.w);
}
template <> __device__ __forceinline__ void unpack<bf16_t>(const uint4& v, float* o) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    o[2 * i] = __uint_as_float(w[i] << 16);
    o[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}
template <> __device__ __forceinline__ void unpack<fp8_t>(const uint4& v, float* o) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w[i] & 0xFFFF), __NV_E4M3);
    __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w[i] >> 16), __NV_E4M3);
    float2 a = __half22float2(*reinterpret_cast<__half2*>(&lo));
    float2 b = __half22float2(*reinterpret_cast<__half2*>(&hi));
    o[4 * i] = a.x; o[4 * i + 1] = a.y; o[4 * i + 2] = b.x; o[4 * i + 3] = b.y;
  }
}

// Scalar load of element i of an activation-typed array (f32 or bf16).
__device__ __forceinline__ float load_act(const void* p, size_t i, int act_f32) {
  return act_f32 ? reinterpret_cast<const float*>(p)[i]
                 : bf16_to_f(reinterpret_cast<const uint16_t*>(p)[i]);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Block-wide sum in a fixed tree order (deterministic). `red` holds >= 32 floats.
__device__ __forceinline__ float block_sum(float v, float* red) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
  v = warp_sum(v);
  __syncthreads();
  if (lane == 0) red[w] = v;
  __syncthreads();
  float t = 0.f;
  if (w == 0) {
    t = lane < nw ? red[lane] : 0.f;
    t = warp_sum(t);
    if (lane == 0) red[0] = t;
  }
  __syncthreads();
  t = red[0];
  __syncthreads();
  return t;
}

// Argmax key of a logit: NaN ranks below every number (like -inf), so every
// argmax here returns a valid index even for a row of NaNs (then the lowest).
__device__ __forceinline__ float am_key(float v) { return v == v ? v : -INFINITY; }

__device__ __forceinline__ float silu(float z) { return z / (1.0f + expf(-z)); }

// Programmatic dependent launch: wait until the preceding kernel in the
// stream has completed and its writes are visible (a no-op when the kernel
// was launched without the attribute), and allow the next kernel to start
// its independent prologue. Every kernel waits in every block before it
// exits, so completion stays transitive along the stream.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Acceptance + commit of sequence slot s of a verify step ("End-to-end OCR
// expert model ...", section 6.1: accept the agreeing prefix from the left,
// the target supplies the token at the first divergence). With g the greedy
// tokens of the K+1 rows: a = max{i <= n_draft : d_j = g_(j-1) for j <= i},
// bonus = g_a. The sequence keeps the KV of its last token and the a accepted
// drafts (length n + a + 1); the rejected rows' slots are stale and are
// overwritten by the next step. Pages wholly past max(new length, reserved
// pages) leave the block table (-1); the host allocator mirrors this.
// Commit of step slot s with a drafts accepted and `bonus` appended.
__device__ __forceinline__ void commit_apply(const Dims& D, const DevState& S, const StepBuf& B, int s, int K, int a,
                                             int bonus) {
  const int max_batch = B.max_batch;
  const int seq = B.step_in[s];
  const int* d = B.step_in + max_batch + s * K;
  const int n = S.seq_len[seq];
  const int new_len = n + a + 1;
  const int no = S.n_out[seq];
  int* out = S.out_tok + (size_t)seq * D.max_ctx;
  for (int j = 0; j < a; ++j)
    if (no + j < D.max_ctx) out[no + j] = d[j];
  if (no + a < D.max_ctx) out[no + a] = bonus;
  S.n_out[seq] = no + a + 1;
  S.seq_len[seq] = new_len;
  S.last_tok[seq] = bonus;
  int keep = (new_len + D.P - 1) / D.P;
  if (S.keep_pages[seq] > keep) keep = S.keep_pages[seq];
  int* bt = const_cast<int*>(S.bt) + (size_t)seq * D.max_pages;
  for (int i = keep; i < D.max_pages; ++i) bt[i] = -1;
  B.step_out[s] = a;
  B.step_out[max_batch + s] = bonus;
  if (s == 0) B.step_out[2 * max_batch] = *S.err;
  int* ua = reinterpret_cast<int*>(B.out_ptrs[0]);
  int* ub = reinterpret_cast<int*>(B.out_ptrs[1]);
  if (ua) ua[s] = a;
  if (ub) ub[s] = bonus;
}

__device__ __forceinline__ void commit_seq(const Dims& D, const DevState& S, const StepBuf& B, int s, int K,
                                           const int* g_rows) {
  const int max_batch = B.max_batch;
  const int* d = B.step_in + max_batch + s * K;
  const int nd = min(max(B.step_in[max_batch + max_batch * K + s], 0), K);
  const int* g = g_rows + s * (K + 1);
  int a = 0;
  while (a < nd && d[a] == g[a]) ++a;
  commit_apply(D, S, B, s, K, a, g[a]);
}

}  // namespace spec
