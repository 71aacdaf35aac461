// Input rows of the FastMTP draft block ("Jina-OCR-v1", section 3.1): for a
// row at position p of depth k,
//   z = P [N_e(E(x_(p+1))) ; N_h(a)],   a = N_o(s),
// where s is the row's source state before the output norm: the decoder's
// final residual of row p (depth 1) or the draft block's output of row p - 1
// at depth k - 1 (k > 1); N_o is the decoder's final RMSNorm (tied), N_e and
// N_h the head's own RMSNorms, E the decoder's embedding (tied), P [h, 2h].
//
//   k_mtp_cat:  one block per row: cat[r] = [N_e(E(tok_r)) ; N_h(N_o(src_r))]
//               (fp32, 2h values); a row whose source pointer is null (padding)
//               gets zeros in its second half; a token -(j + 1) is draft j of
//               the call, read from the device.
//   k_mtp_proj: z[r][o] = sum_j P[o][j] cat[r][j]: one warp per output o, the
//               weight row streamed once for every row of the pass, lanes
//               accumulating in a fixed order and summed by a fixed shuffle
//               tree.
#include "common.cuh"
#include "gemv.cuh"
#include "kernels.h"

namespace spec {

// RMSNorm of n values in shared memory, in place: v * (1 / sqrt(mean(v^2) + eps)) * g.
__device__ __forceinline__ void smem_rmsnorm(float* v, int n, const float* g, float eps, float* red) {
  float ss = 0.f;
  for (int i = threadIdx.x; i < n; i += blockDim.x) ss = fmaf(v[i], v[i], ss);
  const float inv = 1.0f / sqrtf(block_sum(ss, red) / (float)n + eps);
  for (int i = threadIdx.x; i < n; i += blockDim.x) v[i] = (v[i] * inv) * g[i];
  __syncthreads();
}

__global__ void __launch_bounds__(256) k_mtp_cat(Dims D, const int* __restrict__ tok, const float* const* src,
                                                 const int* __restrict__ drafts, const void* tok_embed, const float* __restrict__ enorm,
                                                 const float* __restrict__ final_norm, const float* __restrict__ hnorm,
                                                 float* __restrict__ cat) {
  extern __shared__ __align__(16) float sm[];
  __shared__ float red[32];
  float* e = sm;             // [h]
  float* a = sm + D.h;       // [h]
  const int r = blockIdx.x;
  const int t = tok[r] >= 0 ? tok[r] : drafts[-tok[r] - 1];
  const float* s = src[r];
  for (int i = threadIdx.x; i < D.h; i += blockDim.x) {
    e[i] = load_act(tok_embed, (size_t)t * D.h + i, D.act_f32);
    a[i] = s ? s[i] : 0.f;
  }
  __syncthreads();
  smem_rmsnorm(e, D.h, enorm, D.eps, red);
  if (s) {
    smem_rmsnorm(a, D.h, final_norm, D.eps, red);
    smem_rmsnorm(a, D.h, hnorm, D.eps, red);
  }
  float* out = cat + (size_t)r * 2 * D.h;
  for (int i = threadIdx.x; i < D.h; i += blockDim.x) {
    out[i] = e[i];
    out[D.h + i] = a[i];
  }
}

template <class WT>
__global__ void __launch_bounds__(256) k_mtp_proj(Dims D, const WT* __restrict__ P, const float* __restrict__ cat,
                                                  int n_rows, float* __restrict__ z) {
  constexpr int EP = Elt<WT>::per16;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int o = blockIdx.x * (blockDim.x / 32) + warp;
  if (o >= D.h) return;
  const int K2 = 2 * D.h, nch = K2 / EP;
  const WT* w = P + (size_t)o * K2;
  constexpr int MAXR = 8;
  for (int r0 = 0; r0 < n_rows; r0 += MAXR) {
    const int nr = min(MAXR, n_rows - r0);
    float acc[MAXR];
#pragma unroll
    for (int i = 0; i < MAXR; ++i) acc[i] = 0.f;
    for (int c = lane; c < nch; c += 32) {
      float wv[EP];
      unpack<WT>(ld_stream(w + (size_t)c * EP), wv);
#pragma unroll
      for (int i = 0; i < MAXR; ++i) {
        if (i < nr) {
          const float* x = cat + (size_t)(r0 + i) * K2 + (size_t)c * EP;
#pragma unroll
          for (int q = 0; q < EP; ++q) acc[i] = fmaf(wv[q], x[q], acc[i]);
        }
      }
    }
#pragma unroll
    for (int i = 0; i < MAXR; ++i) {
      if (i < nr) {
        const float v = warp_sum(acc[i]);
        if (lane == 0) z[(size_t)(r0 + i) * D.h + o] = v;
      }
    }
  }
}

void launch_mtp_input(const Dims& D, const int* tok, const float* const* src, const int* drafts, int n_rows,
                      const void* tok_embed,
                      const float* enorm, const float* final_norm, const float* hnorm, const void* P, float* cat,
                      float* z, cudaStream_t st) {
  k_mtp_cat<<<n_rows, 256, 2 * D.h * sizeof(float), st>>>(D, tok, src, drafts, tok_embed, enorm, final_norm, hnorm, cat);
  const int blocks = (D.h + 7) / 8;
  if (D.act_f32) k_mtp_proj<float><<<blocks, 256, 0, st>>>(D, (const float*)P, cat, n_rows, z);
  else k_mtp_proj<bf16_t><<<blocks, 256, 0, st>>>(D, (const bf16_t*)P, cat, n_rows, z);
}

}  // namespace spec
