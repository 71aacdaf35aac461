// Small kernels of the verify step: RoPE tables, row assembly + embedding,
// RMSNorm + router + top-k + token permutation, expert combine, and the
// acceptance / KV-commit kernel.
#include "gemv.cuh"
#include "route.cuh"
#include "kernels.h"

namespace spec {

// cos/sin of p * theta^(-2i/d) for every position and frequency, evaluated in
// double precision and rounded once to fp32.
__global__ void k_rope_table(int max_ctx, int half, int d, double theta, float* cos_t, float* sin_t) {
  const size_t n = (size_t)max_ctx * half;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    const int p = (int)(i / half), j = (int)(i % half);
    const double inv = pow(theta, -(2.0 * j) / (double)d);
    const double a = (double)p * inv;
    cos_t[i] = (float)cos(a);
    sin_t[i] = (float)sin(a);
  }
}

void launch_rope_table(const Dims& D, float* cos_t, float* sin_t, cudaStream_t st) {
  k_rope_table<<<1024, 256, 0, st>>>(D.max_ctx, D.d / 2, D.d, (double)D.theta, cos_t, sin_t);
}

__device__ __forceinline__ void embed_row(const Dims& D, const void* tok_embed, int tok, float* x) {
  for (int k = threadIdx.x; k < D.h; k += blockDim.x) x[k] = load_act(tok_embed, (size_t)tok * D.h + k, D.act_f32);
}

// Verify rows: for sequence slot s of the step, row j holds the last
// committed token (j = 0) or draft j, at position seq_len + j.
__global__ void k_assemble_verify(Dims D, DevState S, StepBuf B, const void* tok_embed, int n_seq, int K) {
  pdl_wait();
  pdl_trigger();
  const int R = K + 1;
  const int row = blockIdx.x, s = row / R, j = row % R;
  const int max_batch = B.max_batch;
  const int seq = B.step_in[s];
  int tok = j == 0 ? S.last_tok[seq] : B.step_in[max_batch + s * K + (j - 1)];
  if (tok < 0 || tok >= D.V) {
    if (threadIdx.x == 0) atomicOr(S.err, DERR_TOKEN);
    tok = 0;
  }
  if (threadIdx.x == 0) {
    B.row_tok[row] = tok;
    B.row_pos[row] = S.seq_len[seq] + j;
    B.row_seq[row] = seq;
  }
  embed_row(D, tok_embed, tok, B.x + (size_t)row * D.h);
}

// Prefill rows: row_src[i] >= 0 is a token id, row_src[i] < 0 selects visual
// row -(row_src[i] + 1) of `vis` (activation storage type).
__global__ void k_assemble_prefill(Dims D, DevState S, StepBuf B, const void* tok_embed, const void* vis,
                                   int seq, int pos0) {
  pdl_wait();
  pdl_trigger();
  const int row = blockIdx.x;
  const int src = B.row_src[row];
  if (threadIdx.x == 0) {
    B.row_tok[row] = src;
    B.row_pos[row] = pos0 + row;
    B.row_seq[row] = seq;
  }
  float* x = B.x + (size_t)row * D.h;
  if (src >= 0) {
    embed_row(D, tok_embed, src, x);
  } else {
    const size_t vr = (size_t)(-(src + 1));
    for (int k = threadIdx.x; k < D.h; k += blockDim.x) x[k] = load_act(vis, vr * D.h + k, D.act_f32);
  }
}

void launch_assemble_verify(const Dims& D, const DevState& S, const StepBuf& B, const void* tok_embed, int n_seq,
                            int K, cudaStream_t st) {
  launch_k(k_assemble_verify, dim3(n_seq * (K + 1)), dim3(256), 0, st, D, S, B, tok_embed, n_seq, K);
}

void launch_assemble_prefill(const Dims& D, const DevState& S, const StepBuf& B, const void* tok_embed,
                             const void* vis, int seq, int pos0, int T, cudaStream_t st) {
  launch_k(k_assemble_prefill, dim3(T), dim3(256), 0, st, D, S, B, tok_embed, vis, seq, pos0);
}

// ---------------------------------------------------------------------------
// FFN input RMSNorm + router + top-k + token permutation. The router
// probabilities are a softmax over all E experts; the top-k are taken in
// (probability desc, id asc) order and used without renormalisation ("Jina AI
// releases jina-ocr-v1", 64 routed + 2 shared experts, top-6). Pair id =
// row * NS + slot (slots 0..k-1 routed, k..k+S-1 shared). Active list:
// routed experts with rows, in id order, then the shared experts with every
// row. The logits come from (row, 16-expert group) blocks; at T <= 8 the
// expert gate/up kernel then runs the top-k and permutation in each block's
// prologue, otherwise the last block of a row takes its top-k and the last
// row builds the permutation. All paths use the same routines in route.cuh,
// so a row's routing does not depend on T.
constexpr int RT_EXPERTS = 16;     // experts per router block (multi-block shape)
constexpr int RT_MAXC = 8;         // 16-byte chunks per lane loaded at once
constexpr int RT_SMALL_T = 8;      // rows handled by the single-block shape

// u = (x * inv) * gamma of one row, into shared (and global when ug != null).
__device__ __forceinline__ void router_u(const float* x, float inv, const float* gamma, int h, float* us,
                                         float* ug) {
  for (int k = threadIdx.x; k < h; k += blockDim.x) {
    const float v = (x[k] * inv) * gamma[k];
    us[k] = v;
    if (ug) ug[k] = v;
  }
}

// Logits of experts e0, e0+1 for nt rows of u (shared, row stride h), by one
// warp: every lane loads all its chunks of both expert rows at once (up to
// 32 * RT_MAXC chunks per pass), then for each row accumulates chunk by chunk
// in increasing order; store(t, ee, logit) receives the warp sums.
template <class RT, class Store>
__device__ __forceinline__ void router_logits2(const RT* Wr, int E, int h, int e0, const float* us, int nt,
                                               Store store) {
  constexpr int EP = Elt<RT>::per16;
  const int lane = threadIdx.x & 31;
  const int nch = h / EP;
  // h <= 32 * RT_MAXC * EP is checked at init, so one pass covers the row
  uint4 wv[2][RT_MAXC];
#pragma unroll
  for (int ee = 0; ee < 2; ++ee)
#pragma unroll
    for (int m = 0; m < RT_MAXC; ++m) {
      const int c = lane + 32 * m;
      wv[ee][m] = (e0 + ee < E && c < nch) ? ld_stream(Wr + (size_t)(e0 + ee) * h + (size_t)c * EP)
                                            : make_uint4(0, 0, 0, 0);
    }
  for (int t = 0; t < nt; ++t) {
    float a0 = 0.f, a1 = 0.f;
    const float* ut = us + (size_t)t * h;
#pragma unroll
    for (int m = 0; m < RT_MAXC; ++m) {
      const int c = lane + 32 * m;
      if (c < nch) {
        float w0[EP], w1[EP];
        unpack<RT>(wv[0][m], w0);
        unpack<RT>(wv[1][m], w1);
#pragma unroll
        for (int i = 0; i < EP; ++i) {
          const float x = ut[c * EP + i];
          a0 = fmaf(w0[i], x, a0);
          a1 = fmaf(w1[i], x, a1);
        }
      }
    }
    a0 = warp_sum(a0);
    a1 = warp_sum(a1);
    store(t, 0, a0);
    store(t, 1, a1);
  }
}

// Logits-only shape (T <= 8): grid (T rows, ceil(E/16) expert groups); each
// block normalises its row (u, written once by group 0) and writes the router
// logits of 16 experts. The expert gate/up kernel then takes the softmax,
// top-k and permutation in its prologue.
template <class RT>
__global__ void __launch_bounds__(256) k_router_logits(Dims D, StepBuf B, const float* __restrict__ gamma,
                                                       const RT* __restrict__ Wr, int T, const float* xres) {
  extern __shared__ __align__(16) float sm[];
  float* us = sm;                 // [h]
  __shared__ float inv[1];
  pdl_wait();
  pdl_trigger();
  const int row = blockIdx.x, grp = blockIdx.y;
  const int warp = threadIdx.x >> 5;
  const float* x = xres + (size_t)row * D.h;
  if (warp == 0) row_inv_rms(x, 1, D.h, D.eps, inv);
  __syncthreads();
  router_u(x, inv[0], gamma, D.h, us, grp == 0 ? B.u + (size_t)row * D.h : nullptr);
  __syncthreads();
  if (D.E > 0) {
    const int e0 = grp * RT_EXPERTS + warp * 2;
    router_logits2<RT>(Wr, D.E, D.h, e0, us, 1, [&](int, int ee, float v) {
      if ((threadIdx.x & 31) == 0 && e0 + ee < D.E) B.rlogit[(size_t)row * D.E + e0 + ee] = v;
    });
  }
}

// Multi-block shape: grid (T rows, ceil(E/16) expert groups).
template <class RT>
__global__ void __launch_bounds__(256) k_router(Dims D, StepBuf B, const float* __restrict__ gamma,
                                                const RT* __restrict__ Wr, int T, const float* xres) {
  extern __shared__ __align__(16) float sm[];
  float* us = sm;                 // [h]
  __shared__ float inv[1];
  __shared__ int s_last;
  pdl_wait();
  pdl_trigger();
  const int row = blockIdx.x, grp = blockIdx.y;
  const int warp = threadIdx.x >> 5;
  const float* x = xres + (size_t)row * D.h;
  if (warp == 0) row_inv_rms(x, 1, D.h, D.eps, inv);
  __syncthreads();
  router_u(x, inv[0], gamma, D.h, us, grp == 0 ? B.u + (size_t)row * D.h : nullptr);
  __syncthreads();
  if (D.E > 0) {
    const int e0 = grp * RT_EXPERTS + warp * 2;
    router_logits2<RT>(Wr, D.E, D.h, e0, us, 1, [&](int, int ee, float v) {
      if ((threadIdx.x & 31) == 0 && e0 + ee < D.E) B.rlogit[(size_t)row * D.E + e0 + ee] = v;
    });
  }
  // ---- the last expert-group block of this row: softmax + top-k ----
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    s_last = (atomicAdd(B.cnt_row + row, 1) == (int)gridDim.y - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  if (D.E > 0 && warp == 0) {
    float* lgs = us;                              // reuse: this row's logits via L2
    for (int e = threadIdx.x; e < D.E; e += 32) lgs[e] = __ldcg(B.rlogit + (size_t)row * D.E + e);
    __syncwarp();
    router_topk(lgs, D.E, D.k, B.ids + row * D.k, B.wts + row * D.k);
  }
  if (threadIdx.x == 0) B.cnt_row[row] = 0;
  // ---- the last row builds the permutation ----
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    s_last = (atomicAdd(B.counter, 1) == (int)gridDim.x - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  int* s_ids = reinterpret_cast<int*>(sm);
  for (int j = threadIdx.x; j < T * D.k; j += blockDim.x) s_ids[j] = __ldcg(B.ids + j);
  __syncthreads();
  router_permute(D, T, s_ids, s_ids + T * D.k, RouteOut{B.act_expert, B.act_off, B.act_cnt, B.n_active, B.perm});
  if (threadIdx.x == 0) *B.counter = 0;
}

cudaError_t configure_small_kernels() {
  cudaError_t e = cudaSuccess, r;
#define ALLOW(k) if ((r = allow_dyn_smem(k)) != cudaSuccess) e = r
  ALLOW(k_router<float>); ALLOW(k_router<bf16_t>);
  ALLOW(k_router_logits<float>); ALLOW(k_router_logits<bf16_t>);
#undef ALLOW
  return e;
}

void launch_router(const Dims& D, const StepBuf& B, const LayerW& W, int T, const float* xres, bool full,
                   cudaStream_t st) {
  const size_t perm_words = (size_t)T * D.k + permute_scratch_words(D.E, T * D.k);
  const dim3 grid(T, D.E > 0 ? (D.E + RT_EXPERTS - 1) / RT_EXPERTS : 1);
  if (!full && T <= RT_SMALL_T) {
    const size_t sm = (size_t)D.h * sizeof(float);
    if (D.act_f32) launch_k(k_router_logits<float>, grid, dim3(256), sm, st, D, B, W.ffn_norm, (const float*)W.w_router, T, xres);
    else launch_k(k_router_logits<bf16_t>, grid, dim3(256), sm, st, D, B, W.ffn_norm, (const bf16_t*)W.w_router, T, xres);
    return;
  }
  const size_t words = (size_t)D.h > perm_words ? (size_t)D.h : perm_words;
  const size_t sm = words * sizeof(float);
  if (D.act_f32) launch_k(k_router<float>, grid, dim3(256), sm, st, D, B, W.ffn_norm, (const float*)W.w_router, T, xres);
  else launch_k(k_router<bf16_t>, grid, dim3(256), sm, st, D, B, W.ffn_norm, (const bf16_t*)W.w_router, T, xres);
}

bool route_in_gateup(int T) { return T <= RT_SMALL_T; }

// ---------------------------------------------------------------------------
// Acceptance + commit as its own kernel (one thread per sequence); the
// verify step normally runs it inside the LM head's last block.
__global__ void k_commit(Dims D, DevState S, StepBuf B, int n_seq, int K) {
  pdl_wait();
  const int s = blockIdx.x * blockDim.x + threadIdx.x;
  if (s < n_seq) commit_seq(D, S, B, s, K, B.g);
}

void launch_commit(const Dims& D, const DevState& S, const StepBuf& B, int n_seq, int K, cudaStream_t st) {
  launch_k(k_commit, dim3((n_seq + 63) / 64), dim3(64), 0, st, D, S, B, n_seq, K);
}

// Commit of a sampled step: the accepted count and appended token come from
// the rejection sampler. A sequence it reports as failed (-1: a draft not a
// token, -2: a wait ran out) raises the matching error bit and is not
// committed.
__global__ void k_commit_sampled(Dims D, DevState S, StepBuf B, int n_seq, int K, const int* __restrict__ acc,
                                 const int* __restrict__ tok) {
  pdl_wait();
  for (int s = threadIdx.x; s < n_seq; s += blockDim.x) {
    const int a = acc[s];
    if (a >= 0) {
      commit_apply(D, S, B, s, K, a, tok[s]);
    } else {
      atomicOr(S.err, a == -2 ? DERR_TIMEOUT : DERR_TOKEN);
      B.step_out[s] = -1;
      B.step_out[B.max_batch + s] = -1;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) B.step_out[2 * B.max_batch] = *reinterpret_cast<volatile int*>(S.err);
}

void launch_commit_sampled(const Dims& D, const DevState& S, const StepBuf& B, int n_seq, int K, const int* acc,
                           const int* tok, cudaStream_t st) {
  launch_k(k_commit_sampled, dim3(1), dim3(256), 0, st, D, S, B, n_seq, K, acc, tok);
}

// Copy device-resident step inputs into the staging block.
__global__ void k_stage_dev(StepBuf B, int n_seq, int K, const int* seq_ids, const int* drafts,
                            const int* n_draft, int* out_acc, int* out_bonus) {
  const int max_batch = B.max_batch;
  if (threadIdx.x == 0) {
    B.out_ptrs[0] = reinterpret_cast<unsigned long long>(out_acc);
    B.out_ptrs[1] = reinterpret_cast<unsigned long long>(out_bonus);
  }
  for (int i = threadIdx.x; i < n_seq; i += blockDim.x) {
    B.step_in[i] = seq_ids[i];
    B.step_in[max_batch + max_batch * K + i] = n_draft[i];
  }
  for (int i = threadIdx.x; i < n_seq * K; i += blockDim.x) B.step_in[max_batch + i] = drafts[i];
}

void launch_stage_dev(const StepBuf& B, int n_seq, int K, const int* seq_ids, const int* drafts,
                      const int* n_draft, int* out_acc, int* out_bonus, cudaStream_t st) {
  k_stage_dev<<<1, 256, 0, st>>>(B, n_seq, K, seq_ids, drafts, n_draft, out_acc, out_bonus);
}

int launches_per_step(const Dims& D, int T) {
  // assemble + per layer (qkv + RoPE + KV write, split-KV attention + merge,
  // O-proj + residual, router + top-k + permute, gate/up + SwiGLU, down,
  // combine) + LM head with argmax and accept/commit
  (void)T;
  return 1 + D.L * 7 + 1;
}

}  // namespace spec
