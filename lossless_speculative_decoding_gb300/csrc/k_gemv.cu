// Final RMSNorm + LM head + greedy argmax for a set of activation rows, with
// per-block candidates reduced by a second kernel (the kernel-level entry
// points spec_lmhead_argmax / spec_lmhead_argmax_noalloc use this form; the
// verify step uses the streaming kernel in k_stream.cu).
#include "gemv.cuh"
#include "kernels.h"

namespace spec {

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
      const float c = am_key(cand[tt][i]);
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
      const float c = am_key(__ldcg(B.am_val + base + i));
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
    const float c = am_key(B.am_val[(size_t)r * B.n_vblocks + i]);
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
  ALLOW(k_lmhead<float>); ALLOW(k_lmhead<bf16_t>);
#undef ALLOW
  return e;
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
