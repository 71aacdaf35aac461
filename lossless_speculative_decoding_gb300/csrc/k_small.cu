// Small kernels of the verify step: RoPE tables, row assembly + embedding,
// RMSNorm + router + top-k + token permutation, expert combine, and the
// acceptance / KV-commit kernel.
#include "common.cuh"
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
// FFN input RMSNorm + router + top-k + token permutation. Grid (T rows,
// ceil(E/16) expert groups): each block normalises its row (u, written once
// by group 0) and computes the router logits of 16 experts, every warp
// issuing all loads of its two expert rows at once. The last group block of a
// row computes that row's softmax over all E experts and its top-k (in
// (probability desc, id asc) order, used without renormalisation: "Jina AI
// releases jina-ocr-v1", 64 routed + 2 shared experts, top-6); the last row
// builds the per-expert pair lists. Pair id = row * NS + slot (slots 0..k-1
// routed, k..k+S-1 shared). Active list: routed experts with rows, in id
// order, then the shared experts with every row.
constexpr int RT_EXPERTS = 16;     // experts per router block
constexpr int RT_MAXC = 8;         // 16-byte chunks per lane loaded at once

template <class RT>
__global__ void __launch_bounds__(256) k_router(Dims D, StepBuf B, const float* __restrict__ gamma,
                                                const RT* __restrict__ Wr, int T) {
  extern __shared__ __align__(16) float sm[];
  float* u = sm;                 // [h]
  __shared__ float red[32];
  __shared__ int s_last;
  pdl_wait();
  pdl_trigger();
  const int row = blockIdx.x, grp = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float* x = B.x + (size_t)row * D.h;
  float ss = 0.f;
  for (int k = threadIdx.x; k < D.h; k += blockDim.x) ss = fmaf(x[k], x[k], ss);
  ss = block_sum(ss, red);
  const float inv = 1.0f / sqrtf(ss / (float)D.h + D.eps);
  for (int k = threadIdx.x; k < D.h; k += blockDim.x) {
    const float v = (x[k] * inv) * gamma[k];
    u[k] = v;
    if (grp == 0) B.u[(size_t)row * D.h + k] = v;
  }
  __syncthreads();
  if (D.E > 0) {
    constexpr int EP = Elt<RT>::per16;
    const int nch = D.h / EP;
    const int e0 = grp * RT_EXPERTS + warp * 2;
    float acc[2] = {0.f, 0.f};
    for (int cb = lane; cb < nch; cb += 32 * RT_MAXC) {
      uint4 wv[2][RT_MAXC];
#pragma unroll
      for (int ee = 0; ee < 2; ++ee)
#pragma unroll
        for (int m = 0; m < RT_MAXC; ++m) {
          const int c = cb + 32 * m;
          wv[ee][m] = (e0 + ee < D.E && c < nch) ? ld_stream(Wr + (size_t)(e0 + ee) * D.h + (size_t)c * EP)
                                                  : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
      for (int ee = 0; ee < 2; ++ee)
#pragma unroll
        for (int m = 0; m < RT_MAXC; ++m) {
          const int c = cb + 32 * m;
          if (c < nch) {
            float w[EP];
            unpack<RT>(wv[ee][m], w);
#pragma unroll
            for (int i = 0; i < EP; ++i) acc[ee] = fmaf(w[i], u[c * EP + i], acc[ee]);
          }
        }
    }
#pragma unroll
    for (int ee = 0; ee < 2; ++ee) {
      const float v = warp_sum(acc[ee]);
      if (lane == 0 && e0 + ee < D.E) B.rlogit[(size_t)row * D.E + e0 + ee] = v;
    }
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
    // softmax over E <= 256 logits, lane l owning experts l, l+32, ...
    constexpr int MAXE = 8;
    float v[MAXE];
    float m = -INFINITY;
#pragma unroll
    for (int i = 0; i < MAXE; ++i) {
      const int e = lane + 32 * i;
      v[i] = e < D.E ? __ldcg(B.rlogit + (size_t)row * D.E + e) : -INFINITY;
      m = fmaxf(m, v[i]);
    }
    m = warp_max(m);
    float z = 0.f;
#pragma unroll
    for (int i = 0; i < MAXE; ++i) {
      v[i] = (lane + 32 * i < D.E) ? expf(v[i] - m) : 0.f;
      z += v[i];
    }
    z = warp_sum(z);
#pragma unroll
    for (int i = 0; i < MAXE; ++i) v[i] = (lane + 32 * i < D.E) ? v[i] / z : -1.f;
    // top-k: k rounds of a warp argmax, (probability desc, id asc)
    for (int r = 0; r < D.k; ++r) {
      float bv = -1.f;
      int bi = 0x7fffffff;
#pragma unroll
      for (int i = 0; i < MAXE; ++i) {
        const int e = lane + 32 * i;
        if (v[i] > bv) { bv = v[i]; bi = e; }      // increasing e: ties keep the lower id
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
      }
      if (lane == 0) {
        B.ids[row * D.k + r] = bi;
        B.wts[row * D.k + r] = bv;
      }
#pragma unroll
      for (int i = 0; i < MAXE; ++i)
        if (lane + 32 * i == bi) v[i] = -1.f;        // taken
    }
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
  const int nk = T * D.k;
  int* s_ids = reinterpret_cast<int*>(sm);        // reuse: [nk] ids, [E] counts, [E] offsets
  int* cnt = s_ids + nk;
  int* offs = cnt + (D.E > 0 ? D.E : 1);
  for (int j = threadIdx.x; j < nk; j += blockDim.x) s_ids[j] = __ldcg(B.ids + j);
  __syncthreads();
  for (int e = threadIdx.x; e < D.E; e += blockDim.x) {
    int c = 0;
    for (int j = 0; j < nk; ++j) c += (s_ids[j] == e);
    cnt[e] = c;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int o = 0, na = 0;
    for (int e = 0; e < D.E; ++e) {
      offs[e] = o;
      if (cnt[e] > 0) {
        B.act_expert[na] = e; B.act_off[na] = o; B.act_cnt[na] = cnt[e];
        ++na;
      }
      o += cnt[e];
    }
    for (int s = 0; s < D.S; ++s) {
      B.act_expert[na] = D.E + s; B.act_off[na] = nk + s * T; B.act_cnt[na] = T;
      ++na;
    }
    *B.n_active = na;
  }
  __syncthreads();
  for (int e = threadIdx.x; e < D.E; e += blockDim.x) {
    if (cnt[e] == 0) continue;
    int c = offs[e];
    for (int j = 0; j < nk; ++j)
      if (s_ids[j] == e) B.perm[c++] = (j / D.k) * D.NS + (j % D.k);
  }
  for (int i = threadIdx.x; i < D.S * T; i += blockDim.x) {
    const int s = i / T, r = i % T;
    B.perm[nk + i] = r * D.NS + D.k + s;
  }
  if (threadIdx.x == 0) *B.counter = 0;
}

cudaError_t configure_small_kernels() {
  cudaError_t e = allow_dyn_smem(k_router<float>);
  cudaError_t f = allow_dyn_smem(k_router<bf16_t>);
  return e != cudaSuccess ? e : f;
}

void launch_router(const Dims& D, const StepBuf& B, const LayerW& W, int T, cudaStream_t st) {
  const int E1 = D.E > 0 ? D.E : 1;
  const size_t words = (size_t)D.h > (size_t)T * D.k + 2 * E1 ? (size_t)D.h : (size_t)T * D.k + 2 * E1;
  const size_t sm = words * sizeof(float);
  const dim3 grid(T, D.E > 0 ? (D.E + RT_EXPERTS - 1) / RT_EXPERTS : 1);
  if (D.act_f32) {
    launch_k(k_router<float>, grid, dim3(256), sm, st, D, B, W.ffn_norm, (const float*)W.w_router, T);
  } else {
    launch_k(k_router<bf16_t>, grid, dim3(256), sm, st, D, B, W.ffn_norm, (const bf16_t*)W.w_router, T);
  }
}

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

int launches_per_step(const Dims& D) {
  // assemble + per layer (qkv + RoPE + KV write, split-KV attention + merge,
  // O-proj + residual, router + top-k + permute, gate/up + SwiGLU, down +
  // combine) + LM head with argmax and accept/commit
  return 1 + D.L * 6 + 1;
}

}  // namespace spec
