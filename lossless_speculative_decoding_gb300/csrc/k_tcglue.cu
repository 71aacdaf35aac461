// Glue kernels around the tensor-core GEMMs (steps with more than 8 rows):
// RMSNorm to the bf16 MMA operand, RoPE + paged KV write from the QKV GEMM's
// fp32 output, gathering routed rows into the expert-permuted bf16 operand,
// and the argmax over the LM head's per-tile candidates followed by the
// accept/commit.
#include "gemv.cuh"
#include "kernels.h"

namespace spec {

// v = (x[t][k] * inv_t) * gamma[k] as operand parts hi, lo and, when out_lo2
// is given, lo2 (split_parts: bf16 parts of v, or with f16 f16 parts of
// 256 v); one block per row. The inverse RMS uses row_inv_rms, the arithmetic
// of every other RMSNorm here.
__global__ void k_norm_bf16(Dims D, const float* __restrict__ x, const float* __restrict__ gamma,
                            uint16_t* __restrict__ out, uint16_t* __restrict__ out_lo, uint16_t* __restrict__ out_lo2,
                            int f16) {
  __shared__ float inv[1];
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.x;
  const float* xr = x + (size_t)t * D.h;
  if (threadIdx.x < 32) row_inv_rms(xr, 1, D.h, D.eps, inv);
  __syncthreads();
  const float s = inv[0];
  for (int k = threadIdx.x; k < D.h; k += blockDim.x) {
    const float v = (xr[k] * s) * gamma[k];
    uint16_t p[3];
    split_parts(v, f16, out_lo2 ? 3 : 2, p);
    out[(size_t)t * D.h + k] = p[0];
    out_lo[(size_t)t * D.h + k] = p[1];
    if (out_lo2) out_lo2[(size_t)t * D.h + k] = p[2];
  }
}

// RoPE on the q and k heads of qkv[t] (fp32, rows q heads | k heads | v heads)
// and the paged write of k and v; q goes to B.q. grid (T, Hq + 2 Hkv), d/2
// threads: thread i handles the rotary pair (i, i + d/2).
__global__ void k_rope_kv(Dims D, DevState S, StepBuf B, int layer) {
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.x, head = blockIdx.y, half = D.d / 2;
  const int pos = B.row_pos[t];
  if (pos < 0 || pos >= D.max_ctx) {
    if (threadIdx.x == 0) atomicOr(S.err, DERR_POS);
    return;
  }
  const int qkv_rows = (D.Hq + 2 * D.Hkv) * D.d;
  const float* src = B.qkv + (size_t)t * qkv_rows + (size_t)head * D.d;
  const bool is_v = head >= D.Hq + D.Hkv;
  int page = -1;
  size_t base = 0;
  if (head >= D.Hq) {
    const int pi = pos / D.P;
    page = pi < D.max_pages ? S.bt[(size_t)B.row_seq[t] * D.max_pages + pi] : -1;
    if (page < 0) {
      if (threadIdx.x == 0) atomicOr(S.err, DERR_PAGE);
      return;
    }
    const int hk = head - D.Hq - (is_v ? D.Hkv : 0);
    base = (size_t)page * D.page_elems + ((((size_t)layer * D.Hkv + hk) * 2 + (is_v ? 1 : 0)) * D.P + (pos % D.P)) * D.d;
  }
  for (int i = threadIdx.x; i < half; i += blockDim.x) {
    const float a = src[i], b = src[i + half];
    float o0 = a, o1 = b;
    if (!is_v) {
      const int rp = B.row_rope ? B.row_rope[t] : pos;
      const float c = S.rope_cos[(size_t)rp * half + i], s = S.rope_sin[(size_t)rp * half + i];
      o0 = a * c - b * s;
      o1 = b * c + a * s;
    }
    if (head < D.Hq) {
      float* q = B.q + ((size_t)t * D.Hq + head) * D.d;
      q[i] = o0;
      q[i + half] = o1;
    } else if (D.act_f32) {
      reinterpret_cast<float*>(S.kv)[base + i] = o0;
      reinterpret_cast<float*>(S.kv)[base + i + half] = o1;
    } else {
      reinterpret_cast<uint16_t*>(S.kv)[base + i] = f_to_bf16(o0);
      reinterpret_cast<uint16_t*>(S.kv)[base + i + half] = f_to_bf16(o1);
    }
  }
}

// xperm[i] = u[perm[i] / NS] as hi + lo operand parts, for the T * NS permuted pairs.
__global__ void k_gather_bf16(Dims D, StepBuf B, int T) {
  pdl_wait();
  pdl_trigger();
  const int i = blockIdx.x;
  if (i >= T * D.NS) return;
  const int row = B.perm[i] / D.NS;
  const float* u = B.u + (size_t)row * D.h;
  for (int k = threadIdx.x; k < D.h; k += blockDim.x) {
    uint16_t p[2];
    split_parts(u[k], D.op_f16, 2, p);
    B.xperm[(size_t)i * D.h + k] = p[0];
    B.xperm_lo[(size_t)i * D.h + k] = p[1];
  }
}

// g[t] = argmax over the per-tile candidates (larger value wins, equal values
// keep the lower index); then, when asked, the accept/commit of the step.
// Greedy token of every row from the GEMM's per-tile candidates (one warp a
// row, lowest index on ties), then, with commit, acceptance and commit by the
// block that finishes last (arrival counter B.counter[1], left at zero).
constexpr int AM_ROWS = 8;                         // rows (warps) per block
__global__ void __launch_bounds__(AM_ROWS * 32) k_argmax_commit(Dims D, DevState S, StepBuf B, int T, int ld,
                                                                 int commit, int n_seq, int K) {
  pdl_wait();
  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.x * AM_ROWS + warp;
  if (row < T) {
    const float* vals = B.am_val + (size_t)row * ld;
    const int* idx = B.am_idx + (size_t)row * ld;
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    for (int i0 = lane; i0 < ld; i0 += 4 * 32) {
      float c[4];
      int ci[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {                // four candidates in flight per lane
        const int i = i0 + 32 * u;
        c[u] = i < ld ? am_key(vals[i]) : -INFINITY;
        ci[u] = i < ld ? idx[i] : 0x7fffffff;
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (c[u] > bv || (c[u] == bv && ci[u] < bi)) { bv = c[u]; bi = ci[u]; }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
    }
    if (lane == 0) B.g[row] = bi;
  }
  if (!commit) return;
  __shared__ int s_last;
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    s_last = atomicAdd(B.counter + 1, 1) == (int)gridDim.x - 1;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const int mb = B.max_batch, R = K + 1;
  for (int s = threadIdx.x; s < n_seq; s += blockDim.x) {
    // the other blocks' tokens, read past L1
    const int* d = B.step_in + mb + s * K;
    const int nd = min(max(B.step_in[mb + mb * K + s], 0), K);
    int a = 0;
    while (a < nd && d[a] == __ldcg(B.g + s * R + a)) ++a;
    commit_apply(D, S, B, s, K, a, __ldcg(B.g + s * R + a));
  }
  if (threadIdx.x == 0) B.counter[1] = 0;
}

void launch_norm_bf16(const Dims& D, const float* x, const float* gamma, uint16_t* out, uint16_t* out_lo,
                      uint16_t* out_lo2, int T, int f16, cudaStream_t st) {
  launch_k(k_norm_bf16, dim3(T), dim3(256), 0, st, D, x, gamma, out, out_lo, out_lo2, f16);
}

void launch_rope_kv(const Dims& D, const DevState& S, const StepBuf& B, int layer, int T, cudaStream_t st) {
  int thr = D.d / 2;
  launch_k(k_rope_kv, dim3(T, D.Hq + 2 * D.Hkv), dim3(thr), 0, st, D, S, B, layer);
}

void launch_gather_bf16(const Dims& D, const StepBuf& B, int T, cudaStream_t st) {
  launch_k(k_gather_bf16, dim3(T * D.NS), dim3(256), 0, st, D, B, T);
}

void launch_argmax_commit(const Dims& D, const DevState& S, const StepBuf& B, int T, int ld, bool commit, int n_seq,
                          int K, cudaStream_t st) {
  launch_k(k_argmax_commit, dim3((T + AM_ROWS - 1) / AM_ROWS), dim3(AM_ROWS * 32), 0, st, D, S, B, T, ld,
           (int)commit, n_seq, K);
}

}  // namespace spec
