// Weight-streaming kernels of the verify step (persistent grids, PDL).
//
// At verify-step sizes every projection reads each weight once and uses it
// for only a few rows, so these kernels are bound by HBM bandwidth and, at
// T = 4 rows, close to the issue limit. Each kernel runs a persistent grid
// (two 256-thread blocks per SM, 128 registers); every warp walks work items
// (4 weight rows x up to TP = 4 activation rows) with a grid stride,
// streaming weights with 16-byte non-allocating loads, accumulating with
// packed fma.rn.f32x2 (even/odd element sums) and reducing the lanes with a
// fixed butterfly. The next item's first weights are loaded before the
// current item's reduction, and -- where the weights do not depend on the
// preceding kernel -- before the programmatic-dependent-launch wait, so the
// fetch overlaps the predecessor's tail.
//
// Fused work: the RMSNorm is applied while staging the QKV / LM-head input
// rows in shared memory; RoPE + the paged KV write after QKV; the residual
// add after the output projection; SwiGLU after gate/up; the argmax (running
// per-warp best, last block reduces) and the accept/commit after the LM head. Every output's arithmetic is independent of T, of the batch
// and of the launch shape, which keeps speculative and greedy decoding
// bit-identical.
#include "gemv.cuh"
#include "kernels.h"
#include "route.cuh"

namespace spec {

constexpr int SG = 3;          // chunk groups in flight per lane
constexpr int SBPS = 2;        // persistent blocks per SM

__host__ __device__ static inline int cdiv(int a, int b) { return (a + b - 1) / b; }

// Shared-memory layout of the kernels that stage normalised input rows:
// [inv: T (padded to 4)][xs: TP x K normalised rows of the current pass].
struct StageLayout {
  int inv, xs, total;   // float offsets / total floats
  __host__ __device__ StageLayout(int T, int K) {
    inv = 0;
    xs = (T + 3) & ~3;
    total = xs + GEMV_TP * K;
  }
};

// ---------------------------------------------------------------------------
// QKV projection + RoPE + paged KV write. Unit = rows {i0, i0+1, i0+d/2,
// i0+1+d/2} of one head (both halves of two rotary pairs in one warp).
template <class WT>
__global__ void __launch_bounds__(256, SBPS) k_qkv_s(Dims D, DevState S, StepBuf B, const float* __restrict__ gamma,
                                                     const WT* __restrict__ W, const float* __restrict__ scale,
                                                     int layer, int T, const float* x) {
  extern __shared__ __align__(16) float sm[];
  const StageLayout Ls(T, D.h);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q4 = D.d / 4, half = D.d / 2;
  const int nunits = (D.Hq + 2 * D.Hkv) * q4;
  const int npass = cdiv(T, GEMV_TP);
  const int stride = gridDim.x * GEMV_WARPS;
  const int nch = D.h / Elt<WT>::per16;
  const int u0 = blockIdx.x * GEMV_WARPS + warp;
  uint4 wv[SG][4];
  const WT* wr[4];
  auto set_rows = [&](int unit) {
    const int base = (unit / q4) * D.d, i0 = 2 * (unit % q4);
    wr[0] = W + (size_t)(base + i0) * D.h;
    wr[1] = W + (size_t)(base + i0 + 1) * D.h;
    wr[2] = W + (size_t)(base + i0 + half) * D.h;
    wr[3] = W + (size_t)(base + i0 + 1 + half) * D.h;
  };
  if (u0 < nunits) {
    set_rows(u0);
    load_group<WT, 4, SG>(wv, wr, nch, lane);
  }
  pdl_wait();
  pdl_trigger();
  float* inv = sm + Ls.inv;
  float* xs = sm + Ls.xs;
  row_inv_rms(x, T, D.h, D.eps, inv);
  __syncthreads();
  for (int pass = 0; pass < npass; ++pass) {
    const int t0 = pass * GEMV_TP, nvalid = min(GEMV_TP, T - t0);
    if (pass > 0) __syncthreads();
    stage_norm(xs, x, t0, nvalid, D.h, inv, gamma);
    __syncthreads();
    const float* xr[GEMV_TP];
#pragma unroll
    for (int t = 0; t < GEMV_TP; ++t) xr[t] = xs + t * D.h;
    for (int unit = u0; unit < nunits; unit += stride) {
      const int head = unit / q4, i0 = 2 * (unit % q4), base = head * D.d;
      float acc[16];
      unit_dot2<WT, 4, GEMV_TP, SG>(wv, wr, D.h, xr, acc);
      const int nx = unit + stride < nunits ? unit + stride : (pass + 1 < npass ? u0 : -1);
      if (nx >= 0) {
        set_rows(nx);
        load_group<WT, 4, SG>(wv, wr, nch, lane);
      }
      const float sum = reduce_scatter<16>(acc);
      const int v = (lane >> 1) & 15, r = v / GEMV_TP, t = v % GEMV_TP;
      const int rowW = base + i0 + (r & 1) + (r >= 2 ? half : 0);
      const float val = scale != nullptr ? sum * scale[rowW] : sum;
      const int pv = ((r ^ 2) * GEMV_TP + t) * 2;          // lane holding the rotary partner
      const float partner = __shfl_sync(0xffffffffu, val, pv);
      if ((lane & 1) || t >= nvalid) continue;
      const int row = t0 + t;
      const int pos = B.row_pos[row];
      if (pos < 0 || pos >= D.max_ctx) { atomicOr(S.err, DERR_POS); continue; }
      const int j = i0 + (r & 1);                           // rotary frequency index
      const int dim = (r < 2) ? j : j + half;
      float outv = val;
      if (head < D.Hq + D.Hkv) {
        const int rp = B.row_rope ? B.row_rope[row] : pos;
        const float c = S.rope_cos[(size_t)rp * half + j], s = S.rope_sin[(size_t)rp * half + j];
        // first half: a cos - b sin; second half: b cos + a sin (a = first-half value)
        outv = (r < 2) ? (val * c - partner * s) : (val * c + partner * s);
      }
      if (head < D.Hq) {
        B.q[((size_t)row * D.Hq + head) * D.d + dim] = outv;
        continue;
      }
      const int is_v = head >= D.Hq + D.Hkv;
      const int hk = head - D.Hq - (is_v ? D.Hkv : 0);
      const int seq = B.row_seq[row];
      const int pi = pos / D.P;
      const int page = pi < D.max_pages ? S.bt[(size_t)seq * D.max_pages + pi] : -1;
      if (page < 0) { atomicOr(S.err, DERR_PAGE); continue; }
      const size_t off = (size_t)page * D.page_elems +
                         ((((size_t)layer * D.Hkv + hk) * 2 + is_v) * D.P + (pos % D.P)) * D.d + dim;
      if (D.act_f32) reinterpret_cast<float*>(S.kv)[off] = outv;
      else reinterpret_cast<uint16_t*>(S.kv)[off] = f_to_bf16(outv);
    }
  }
}

// ---------------------------------------------------------------------------
// Output projection + residual: x[t][o] += sum_k W_o[o][k] * attn[t][k].
template <class WT>
__global__ void __launch_bounds__(256, SBPS) k_oproj_s(Dims D, StepBuf B, const WT* __restrict__ W,
                                                       const float* __restrict__ scale, int T, float* xres) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int K = D.Hq * D.d;
  const int npass = cdiv(T, GEMV_TP);
  const int nitems = (D.h / 4) * npass;
  const int stride = gridDim.x * GEMV_WARPS;
  const int nch = K / Elt<WT>::per16;
  int it = blockIdx.x * GEMV_WARPS + warp;
  uint4 wv[SG][4];
  const WT* wr[4];
  auto set_rows = [&](int item) {
    const int o0 = (item / npass) * 4;
#pragma unroll
    for (int r = 0; r < 4; ++r) wr[r] = W + (size_t)(o0 + r) * K;
  };
  if (it < nitems) {
    set_rows(it);
    load_group<WT, 4, SG>(wv, wr, nch, lane);
  }
  pdl_wait();
  pdl_trigger();
  for (; it < nitems; it += stride) {
    const int o0 = (it / npass) * 4, pass = it % npass;
    const int t0 = pass * GEMV_TP, nvalid = min(GEMV_TP, T - t0);
    const float* xr[GEMV_TP];
#pragma unroll
    for (int t = 0; t < GEMV_TP; ++t) xr[t] = t < nvalid ? B.o + (size_t)(t0 + t) * K : nullptr;
    float acc[16];
    unit_dot2<WT, 4, GEMV_TP, SG>(wv, wr, K, xr, acc);
    if (it + stride < nitems) {
      set_rows(it + stride);
      load_group<WT, 4, SG>(wv, wr, nch, lane);
    }
    const float sum = reduce_scatter<16>(acc);
    const int v = (lane >> 1) & 15, r = v / GEMV_TP, t = v % GEMV_TP;
    if ((lane & 1) || t >= nvalid) continue;
    const int o = o0 + r;
    xres[(size_t)(t0 + t) * D.h + o] += scale != nullptr ? sum * scale[o] : sum;
  }
}

// ---------------------------------------------------------------------------
// Active-expert list held in shared memory by the expert kernels:
// [expert][offset][count] per active slot, the pair permutation, the count.
struct ActCache {
  int* ex;
  int* off;
  int* cnt;
  int* perm;
  int* nact;
  __device__ ActCache(int* smi, int max_active, int npairs) {
    ex = smi;
    off = smi + max_active;
    cnt = smi + 2 * max_active;
    perm = smi + 3 * max_active;
    nact = perm + npairs;
  }
  static __host__ __device__ int words(int max_active, int npairs) { return 3 * max_active + npairs + 1; }
};

__device__ __forceinline__ void copy_active(const StepBuf& B, const ActCache& A, int max_active, int npairs) {
  const int n = min(*B.n_active, max_active);
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    A.ex[i] = B.act_expert[i];
    A.off[i] = B.act_off[i];
    A.cnt[i] = B.act_cnt[i];
  }
  for (int i = threadIdx.x; i < npairs; i += blockDim.x) A.perm[i] = B.perm[i];
  if (threadIdx.x == 0) *A.nact = n;
  __syncthreads();
}

// Routing in the gate/up prologue (T <= 8): top-k of every row from the
// router logits, then the permutation, all in shared memory; block 0
// publishes ids/weights (for the combine) and the active list (for down).
__device__ __forceinline__ void route_in_block(const Dims& D, const StepBuf& B, const ActCache& A, int T,
                                               float* lg, int* ids, float* wts, int* scratch) {
  const int warp = threadIdx.x >> 5;
  if (D.E > 0) {
    for (int i = threadIdx.x; i < T * D.E; i += blockDim.x) lg[i] = B.rlogit[i];
    __syncthreads();
    for (int t = warp; t < T; t += blockDim.x / 32) router_topk(lg + t * D.E, D.E, D.k, ids + t * D.k, wts + t * D.k);
    __syncthreads();
  }
  router_permute(D, T, ids, scratch, RouteOut{A.ex, A.off, A.cnt, A.nact, A.perm});
  if (blockIdx.x == 0) {
    for (int i = threadIdx.x; i < T * D.k; i += blockDim.x) {
      B.ids[i] = ids[i];
      B.wts[i] = wts[i];
    }
    const int n = *A.nact;
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
      B.act_expert[i] = A.ex[i];
      B.act_off[i] = A.off[i];
      B.act_cnt[i] = A.cnt[i];
    }
    for (int i = threadIdx.x; i < T * D.NS; i += blockDim.x) B.perm[i] = A.perm[i];
    if (threadIdx.x == 0) *B.n_active = n;
  }
}

// Shared-memory words of the gate/up kernel: active list (+ routing scratch).
__host__ __device__ inline int gateup_words(const Dims& D, int T, int max_active, bool route) {
  int w = ActCache::words(max_active, T * D.NS);
  if (route) w += T * D.E + 2 * T * D.k + permute_scratch_words(D.E, T * D.k);
  return w;
}

// Expert gate/up + SwiGLU. Items: (active-expert slot, output rows j, j+1,
// pass over the slot's routed pairs); the unit streams gate rows j, j+1 and
// up rows j, j+1 and writes h_act[pair][j] = silu(gate) * up. Slots 0..S-1
// are the shared experts, so a warp whose first item is a shared-expert item
// starts streaming its weights before the kernel waits for the router.
template <class WT>
__global__ void __launch_bounds__(256, SBPS) k_gateup_s(Dims D, StepBuf B, const WT* __restrict__ Wg,
                                                        const float* __restrict__ sg, const WT* __restrict__ Wu,
                                                        const float* __restrict__ su, int T, int max_active,
                                                        int route) {
  extern __shared__ __align__(16) int smi[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int npass = cdiv(T, GEMV_TP);
  const int upe = D.inter / 2;
  const int per_slot = upe * npass;
  const int nch = D.h / Elt<WT>::per16;
  const int stride = gridDim.x * GEMV_WARPS;
  const ActCache A(smi, max_active, T * D.NS);
  uint4 wv[SG][4];
  const WT* wr[4];
  auto set_rows_e = [&](int e, int it) {
    const int j = ((it % per_slot) / npass) * 2;
    const size_t eb = (size_t)e * D.inter * D.h;
    wr[0] = Wg + eb + (size_t)j * D.h;
    wr[1] = Wg + eb + (size_t)(j + 1) * D.h;
    wr[2] = Wu + eb + (size_t)j * D.h;
    wr[3] = Wu + eb + (size_t)(j + 1) * D.h;
  };
  const int it0 = blockIdx.x * GEMV_WARPS + warp;
  const bool pre = it0 < D.S * per_slot;             // shared-expert item: expert known now
  if (pre) {
    set_rows_e(D.E + it0 / per_slot, it0);
    load_group<WT, 4, SG>(wv, wr, nch, lane);
  }
  pdl_wait();
  pdl_trigger();
  if (route) {
    float* lg = reinterpret_cast<float*>(smi + ActCache::words(max_active, T * D.NS));
    int* ids = reinterpret_cast<int*>(lg + T * D.E);
    float* wts = reinterpret_cast<float*>(ids + T * D.k);
    int* scratch = reinterpret_cast<int*>(wts + T * D.k);
    route_in_block(D, B, A, T, lg, ids, wts, scratch);
  } else {
    copy_active(B, A, max_active, T * D.NS);
  }
  const int nitems = *A.nact * per_slot;
  auto valid = [&](int it) { return ((it % per_slot) % npass) * GEMV_TP < A.cnt[it / per_slot]; };
  auto next_valid = [&](int it) {
    while (it < nitems && !valid(it)) it += stride;
    return it;
  };
  int it = next_valid(it0);
  if (it < nitems && !(pre && it == it0)) {
    set_rows_e(A.ex[it / per_slot], it);
    load_group<WT, 4, SG>(wv, wr, nch, lane);
  }
  while (it < nitems) {
    const int slot = it / per_slot, rem = it % per_slot;
    const int j = (rem / npass) * 2, p0 = (rem % npass) * GEMV_TP;
    const int e = A.ex[slot];
    const int nvalid = min(GEMV_TP, A.cnt[slot] - p0);
    const int* pairs = A.perm + A.off[slot] + p0;
    int pr[GEMV_TP];
    const float* xr[GEMV_TP];
#pragma unroll
    for (int t = 0; t < GEMV_TP; ++t) {
      pr[t] = t < nvalid ? pairs[t] : 0;
      xr[t] = t < nvalid ? B.u + (size_t)(pr[t] / D.NS) * D.h : nullptr;
    }
    float acc[16];
    unit_dot2<WT, 4, GEMV_TP, SG>(wv, wr, D.h, xr, acc);
    const int nx = next_valid(it + stride);
    if (nx < nitems) {
      set_rows_e(A.ex[nx / per_slot], nx);
      load_group<WT, 4, SG>(wv, wr, nch, lane);
    }
    const float sum = reduce_scatter<16>(acc);          // lane >> 1 = r*TP + t; r: gate j, gate j+1, up j, up j+1
    const float up = __shfl_sync(0xffffffffu, sum, (lane + 2 * 2 * GEMV_TP) & 31);
    const int v = (lane >> 1) & 15, r = v / GEMV_TP, t = v % GEMV_TP;
    if (!(lane & 1) && r < 2 && t < nvalid) {
      const int jj = j + r;
      float g = sum, uu = up;
      if (sg != nullptr) { g *= sg[(size_t)e * D.inter + jj]; uu *= su[(size_t)e * D.inter + jj]; }
      B.h_act[(size_t)pr[t] * D.inter + jj] = silu(g) * uu;
    }
    it = nx;
  }
}

// ---------------------------------------------------------------------------
// Expert down projection y[pair][o] = sum_j W_d[e][o][j] * h_act[pair][j];
// k_combine then adds the slots into the residual.
template <class WT>
__global__ void __launch_bounds__(256, SBPS) k_down_s(Dims D, StepBuf B, const WT* __restrict__ Wd,
                                                      const float* __restrict__ sd, int T, int max_active) {
  extern __shared__ __align__(16) int smi[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int npass = cdiv(T, GEMV_TP);
  const int upe = D.h / 4;
  const int per_slot = upe * npass;
  const int nch = D.inter / Elt<WT>::per16;
  const int stride = gridDim.x * GEMV_WARPS;
  const ActCache A(smi, max_active, T * D.NS);
  uint4 wv[SG][4];
  const WT* wr[4];
  auto set_rows_e = [&](int e, int it) {
    const int o0 = ((it % per_slot) / npass) * 4;
#pragma unroll
    for (int r = 0; r < 4; ++r) wr[r] = Wd + ((size_t)e * D.h + o0 + r) * D.inter;
  };
  const int it0 = blockIdx.x * GEMV_WARPS + warp;
  const bool pre = it0 < D.S * per_slot;             // shared-expert item: expert known now
  if (pre) {
    set_rows_e(D.E + it0 / per_slot, it0);
    load_group<WT, 4, SG>(wv, wr, nch, lane);
  }
  pdl_wait();
  pdl_trigger();
  copy_active(B, A, max_active, T * D.NS);
  const int nitems = *A.nact * per_slot;
  auto valid = [&](int it) { return ((it % per_slot) % npass) * GEMV_TP < A.cnt[it / per_slot]; };
  auto next_valid = [&](int it) {
    while (it < nitems && !valid(it)) it += stride;
    return it;
  };
  int it = next_valid(it0);
  if (it < nitems && !(pre && it == it0)) {
    set_rows_e(A.ex[it / per_slot], it);
    load_group<WT, 4, SG>(wv, wr, nch, lane);
  }
  while (it < nitems) {
    const int slot = it / per_slot, rem = it % per_slot;
    const int o0 = (rem / npass) * 4, p0 = (rem % npass) * GEMV_TP;
    const int e = A.ex[slot];
    const int nvalid = min(GEMV_TP, A.cnt[slot] - p0);
    const int* pairs = A.perm + A.off[slot] + p0;
    int pr[GEMV_TP];
    const float* xr[GEMV_TP];
#pragma unroll
    for (int t = 0; t < GEMV_TP; ++t) {
      pr[t] = t < nvalid ? pairs[t] : 0;
      xr[t] = t < nvalid ? B.h_act + (size_t)pr[t] * D.inter : nullptr;
    }
    float acc[16];
    unit_dot2<WT, 4, GEMV_TP, SG>(wv, wr, D.inter, xr, acc);
    const int nx = next_valid(it + stride);
    if (nx < nitems) {
      set_rows_e(A.ex[nx / per_slot], nx);
      load_group<WT, 4, SG>(wv, wr, nch, lane);
    }
    const float sum = reduce_scatter<16>(acc);
    const int v = (lane >> 1) & 15, r = v / GEMV_TP, t = v % GEMV_TP;
    if (!(lane & 1) && t < nvalid) {
      const int o = o0 + r;
      B.y[(size_t)pr[t] * D.h + o] = sd != nullptr ? sum * sd[(size_t)e * D.h + o] : sum;
    }
    it = nx;
  }
}

// Expert combine, in place: x[t][k] += sum over slots s (in order) of
// w[t][s] * y[t*NS + s][k] (routed weight p, shared weight 1): a = 0, then
// a = fma(w_s, y_s, a) slot by slot, then x + a. A thread takes four
// consecutive columns of one row and loads all of its slots' values before
// the first sum (up to COMB_MAXS slots; more slots take the scalar loop).
constexpr int COMB_MAXS = 16;
__global__ void k_combine(Dims D, StepBuf B, float* x, int T) {
  pdl_wait();
  pdl_trigger();
  const int h4 = D.h / 4, n4 = T * h4;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += gridDim.x * blockDim.x) {
    const int t = i / h4, k4 = i % h4;
    if (D.NS > COMB_MAXS) {
      for (int c = 0; c < 4; ++c) x[(size_t)t * D.h + 4 * k4 + c] = combine_one(x, B.y, B.wts, t, 4 * k4 + c, D.h, D.NS, D.k);
      continue;
    }
    float4 yv[COMB_MAXS];
    float wv[COMB_MAXS];
#pragma unroll
    for (int s = 0; s < COMB_MAXS; ++s) {
      if (s < D.NS) {
        yv[s] = reinterpret_cast<const float4*>(B.y + ((size_t)t * D.NS + s) * D.h)[k4];
        wv[s] = s < D.k ? B.wts[t * D.k + s] : 1.f;
      }
    }
    float4 xv = reinterpret_cast<const float4*>(x + (size_t)t * D.h)[k4];
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
    for (int s = 0; s < COMB_MAXS; ++s) {
      if (s < D.NS) {
        a0 = fmaf(wv[s], yv[s].x, a0);
        a1 = fmaf(wv[s], yv[s].y, a1);
        a2 = fmaf(wv[s], yv[s].z, a2);
        a3 = fmaf(wv[s], yv[s].w, a3);
      }
    }
    xv.x += a0; xv.y += a1; xv.z += a2; xv.w += a3;
    reinterpret_cast<float4*>(x + (size_t)t * D.h)[k4] = xv;
  }
}

// ---------------------------------------------------------------------------
// Final RMSNorm + LM head + greedy argmax (+ accept/commit). Each warp keeps
// the running best (value, index) of its vocabulary rows for every activation
// row of a pass (strict '>' over increasing indices keeps the lowest index on
// ties); the candidates of all warps are reduced by the last block, which then
// commits the step's sequences when asked to.
template <class WT>
__global__ void __launch_bounds__(256, SBPS) k_lmhead_s(Dims D, DevState S, StepBuf B, const WT* __restrict__ W,
                                                        const float* __restrict__ gamma, const float* x, int T,
                                                        float* __restrict__ logits_dbg, int commit, int n_seq,
                                                        int K) {
  extern __shared__ __align__(16) float sm[];
  __shared__ int s_last;
  const StageLayout Ls(T, D.h);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gw = blockIdx.x * GEMV_WARPS + warp;
  const int nw = gridDim.x * GEMV_WARPS;
  const int nunits = D.V / 4;
  const int nch = D.h / Elt<WT>::per16;
  const int npass = cdiv(T, GEMV_TP);
  uint4 wv[SG][4];
  const WT* wr[4];
  auto set_rows = [&](int u) {
#pragma unroll
    for (int r = 0; r < 4; ++r) wr[r] = W + (size_t)(u * 4 + r) * D.h;
  };
  if (gw < nunits) {
    set_rows(gw);
    load_group<WT, 4, SG>(wv, wr, nch, lane);
  }
  pdl_wait();
  pdl_trigger();
  float* inv = sm + Ls.inv;
  float* xs = sm + Ls.xs;
  row_inv_rms(x, T, D.h, D.eps, inv);
  __syncthreads();
  const int v = (lane >> 1) & 15, r = v / GEMV_TP, t = v % GEMV_TP;
  for (int pass = 0; pass < npass; ++pass) {
    const int t0 = pass * GEMV_TP, nvalid = min(GEMV_TP, T - t0);
    if (pass > 0) __syncthreads();
    stage_norm(xs, x, t0, nvalid, D.h, inv, gamma);
    __syncthreads();
    const float* xr[GEMV_TP];
#pragma unroll
    for (int tt = 0; tt < GEMV_TP; ++tt) xr[tt] = xs + tt * D.h;
    float best = -INFINITY;
    int bidx = 0x7fffffff;
    for (int u = gw; u < nunits; u += nw) {
      float acc[16];
      unit_dot2<WT, 4, GEMV_TP, SG>(wv, wr, D.h, xr, acc);
      const int un = u + nw < nunits ? u + nw : (pass + 1 < npass ? gw : -1);
      if (un >= 0) {
        set_rows(un);
        load_group<WT, 4, SG>(wv, wr, nch, lane);
      }
      const float val = reduce_scatter<16>(acc);
      const int vi = u * 4 + r;
      if (logits_dbg != nullptr && !(lane & 1) && t < nvalid) logits_dbg[(size_t)(t0 + t) * D.V + vi] = val;
      const float kv = am_key(val);
      if (kv > best || (kv == best && vi < bidx)) { best = kv; bidx = vi; }
    }
    // combine the four row lanes (r in lane bits 3..4) of each activation row t
#pragma unroll
    for (int o = 8; o <= 16; o <<= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, best, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bidx, o);
      if (ov > best || (ov == best && oi < bidx)) { best = ov; bidx = oi; }
    }
    if (lane < 2 * GEMV_TP && !(lane & 1) && t < nvalid) {
      B.am_val[(size_t)(t0 + t) * B.n_vblocks + gw] = best;
      B.am_idx[(size_t)(t0 + t) * B.n_vblocks + gw] = bidx;
    }
  }
  // the last block reduces every warp's candidates (larger value wins, equal
  // values keep the lower index) and then commits
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    s_last = (atomicAdd(B.cnt_lm, 1) == (int)gridDim.x - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  for (int row = warp; row < T; row += GEMV_WARPS) {
    const size_t base = (size_t)row * B.n_vblocks;
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    for (int i = lane; i < nw; i += 32) {
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
    if (lane == 0) B.g[row] = bi;
  }
  if (threadIdx.x == 0) *B.cnt_lm = 0;
  if (!commit) return;
  __syncthreads();
  __threadfence();
  for (int s = threadIdx.x; s < n_seq; s += blockDim.x) commit_seq(D, S, B, s, K, B.g);
}

// ===========================================================================
// Tensor-core forms (bf16 / e4m3 weights): a block takes one unit of 16
// weight rows at a time against up to 8 columns through mma.sync, its 8
// warps splitting the unit's K steps (mma_part), and block_sum4 adds the
// warps' parts in a fixed order for warp 0, which runs the epilogue. A warp's
// loads of its K slice are all in flight at once, and the next unit's loads
// are issued before the current unit's reduction. Columns are activation rows
// (tokens) or, in the expert kernels, routed pairs; more than 8 (a prefill
// chunk) are taken in passes of 8 over the same weights.
constexpr int MNB = 5;           // K steps per warp in flight
constexpr int MC = 8;            // columns per pass

// normalised rows [t0, t0 + n) of x into xs[MC][K + 4] (zeros past n); the
// 4-float pad keeps the lanes' float4 reads on distinct banks
__device__ __forceinline__ void stage_cols(float* xs, const float* x, int t0, int n, int K, const float* inv,
                                           const float* gamma) {
  const int K4 = K / 4, ld4 = K4 + 1;
  for (int i = threadIdx.x; i < MC * K4; i += blockDim.x) {
    const int t = i / K4, k4 = i % K4;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (t < n) {
      v = reinterpret_cast<const float4*>(x + (size_t)(t0 + t) * K)[k4];
      if (gamma != nullptr) {
        const float sc = inv[t0 + t];
        const float4 g = reinterpret_cast<const float4*>(gamma)[k4];
        v = make_float4((v.x * sc) * g.x, (v.y * sc) * g.y, (v.z * sc) * g.z, (v.w * sc) * g.w);
      }
    }
    reinterpret_cast<float4*>(xs)[t * ld4 + k4] = v;
  }
}

// QKV + RoPE + paged KV write. Unit = rows i0..i0+7 (first half of a head)
// and i0+d/2..i0+d/2+7 (their rotary partners): lane (g, q) of warp 0 holds
// both values of rotary pair i0 + g for columns 2q, 2q+1.
template <class WT>
__global__ void __launch_bounds__(256, SBPS) k_qkv_m(Dims D, DevState S, StepBuf B, const float* __restrict__ gamma,
                                                     const WT* __restrict__ W, const float* __restrict__ scale,
                                                     int layer, int T, const float* x) {
  extern __shared__ __align__(16) float sm[];
  __shared__ float4 red[512];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
  const int half = D.d / 2, upu = half / 8;
  const int nunits = (D.Hq + 2 * D.Hkv) * upu;
  const int npass = cdiv(T, MC);
  float* inv = sm;
  float* xs = sm + ((T + 3) & ~3);
  uint4 va[MNB], vb[MNB];
  Q4Scales<MNB> qs;
  const WT *wlo = W, *whi = W;
  const int nrows = (D.Hq + 2 * D.Hkv) * D.d;
  auto set_rows = [&](int unit) {
    const int base = (unit / upu) * D.d + (unit % upu) * 8 + g;
    wlo = stack_row(W, 0, nrows, base, D.h, &qs.lo);
    whi = stack_row(W, 0, nrows, base + half, D.h, &qs.hi);
  };
  if ((int)blockIdx.x < nunits) {
    set_rows(blockIdx.x);
    mma_load_batch<WT, MNB>(va, vb, wlo, whi, D.h, warp, qs);
  }
  pdl_wait();
  pdl_trigger();
  row_inv_rms(x, T, D.h, D.eps, inv);
  __syncthreads();
  int par = 0;
  for (int pass = 0; pass < npass; ++pass) {
    const int t0 = pass * MC, nvalid = min(MC, T - t0);
    if (pass > 0) __syncthreads();
    stage_cols(xs, x, t0, nvalid, D.h, inv, gamma);
    __syncthreads();
    for (int unit = blockIdx.x; unit < nunits; unit += gridDim.x) {
      const int head = unit / upu, j = (unit % upu) * 8 + g;       // rotary frequency index
      float c[4];
      // three activation parts: the K/V outputs are rounded to bf16 for the
      // cache, and a two-part split would move some of them across a rounding
      // boundary that the exact product does not cross
      mma_part<WT, MNB, 3>(va, vb, wlo, whi, D.h, g < nvalid ? xs + g * (D.h + 4) : nullptr, c, qs);
      const int nx = unit + (int)gridDim.x < nunits ? unit + gridDim.x : (pass + 1 < npass ? (int)blockIdx.x : -1);
      if (nx >= 0) {
        set_rows(nx);
        mma_load_batch<WT, MNB>(va, vb, wlo, whi, D.h, warp, qs);
      }
      block_sum4(c, red, par);
      par ^= 1;
      if (warp != 0) continue;
      float a[2] = {c[0], c[1]}, b[2] = {c[2], c[3]};            // first / second half, columns 2q, 2q+1
      if constexpr (IsQ4<WT>::v) {                                // nvfp4: the matrix's tensor scale
        const float ts = scale[0] * (1.0f / F16_OP_SCALE);
        a[0] *= ts; a[1] *= ts; b[0] *= ts; b[1] *= ts;
      } else if (scale != nullptr) {
        const float sa = scale[head * D.d + j], sb = scale[head * D.d + j + half];
        a[0] *= sa; a[1] *= sa; b[0] *= sb; b[1] *= sb;
      }
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int col = 2 * q + e;
        if (col >= nvalid) continue;
        const int row = t0 + col;
        const int pos = B.row_pos[row];
        if (pos < 0 || pos >= D.max_ctx) { atomicOr(S.err, DERR_POS); continue; }
        float o0 = a[e], o1 = b[e];
        if (head < D.Hq + D.Hkv) {
          const int rp = B.row_rope ? B.row_rope[row] : pos;
          const float cs = S.rope_cos[(size_t)rp * half + j], sn = S.rope_sin[(size_t)rp * half + j];
          o0 = a[e] * cs - b[e] * sn;
          o1 = b[e] * cs + a[e] * sn;
        }
        if (head < D.Hq) {
          float* qd = B.q + ((size_t)row * D.Hq + head) * D.d;
          qd[j] = o0;
          qd[j + half] = o1;
          continue;
        }
        const int is_v = head >= D.Hq + D.Hkv;
        const int hk = head - D.Hq - (is_v ? D.Hkv : 0);
        const int pi = pos / D.P;
        const int page = pi < D.max_pages ? S.bt[(size_t)B.row_seq[row] * D.max_pages + pi] : -1;
        if (page < 0) { atomicOr(S.err, DERR_PAGE); continue; }
        const size_t off = (size_t)page * D.page_elems +
                           ((((size_t)layer * D.Hkv + hk) * 2 + is_v) * D.P + (pos % D.P)) * D.d + j;
        reinterpret_cast<uint16_t*>(S.kv)[off] = f_to_bf16(o0);
        reinterpret_cast<uint16_t*>(S.kv)[off + half] = f_to_bf16(o1);
      }
    }
  }
}

// Output projection + residual: x[t][o] += sum_k W_o[o][k] * attn[t][k].
template <class WT>
__global__ void __launch_bounds__(256, SBPS) k_oproj_m(Dims D, StepBuf B, const WT* __restrict__ W,
                                                       const float* __restrict__ scale, int T, float* xres) {
  __shared__ float4 red[512];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
  const int K = D.Hq * D.d;
  const int npass = cdiv(T, MC);
  const int nitems = (D.h / 16) * npass;
  uint4 va[MNB], vb[MNB];
  Q4Scales<MNB> qs;
  const WT *wlo = W, *whi = W;
  auto set_rows = [&](int item) {
    const int o = (item / npass) * 16 + g;
    wlo = stack_row(W, 0, D.h, o, K, &qs.lo);
    whi = stack_row(W, 0, D.h, o + 8, K, &qs.hi);
  };
  int it = blockIdx.x;
  if (it < nitems) {
    set_rows(it);
    mma_load_batch<WT, MNB>(va, vb, wlo, whi, K, warp, qs);
  }
  pdl_wait();
  pdl_trigger();
  int par = 0;
  for (; it < nitems; it += gridDim.x) {
    const int o = (it / npass) * 16 + g, t0 = (it % npass) * MC, nvalid = min(MC, T - t0);
    float c[4];
    mma_part<WT, MNB>(va, vb, wlo, whi, K, g < nvalid ? B.o + (size_t)(t0 + g) * K : nullptr, c, qs);
    if (it + (int)gridDim.x < nitems) {
      set_rows(it + gridDim.x);
      mma_load_batch<WT, MNB>(va, vb, wlo, whi, K, warp, qs);
    }
    block_sum4(c, red, par);
    par ^= 1;
    if (warp != 0) continue;
    float s0 = 1.f, s1 = 1.f;
    if constexpr (IsQ4<WT>::v) s0 = s1 = scale[0] * (1.0f / F16_OP_SCALE);
    else if (scale != nullptr) { s0 = scale[o]; s1 = scale[o + 8]; }
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int col = 2 * q + e;
      if (col >= nvalid) continue;
      float* xr = xres + (size_t)(t0 + col) * D.h;
      xr[o] += c[e] * s0;
      xr[o + 8] += c[2 + e] * s1;
    }
  }
}

// Expert gate/up + SwiGLU. Items: (active slot, gate/up rows j..j+7, pass of
// 8 routed pairs); lanes of warp 0 hold gate row j+g and up row j+g of their
// columns.
template <class WT>
__global__ void __launch_bounds__(256, SBPS) k_gateup_m(Dims D, StepBuf B, const WT* __restrict__ Wg,
                                                        const float* __restrict__ sg, const WT* __restrict__ Wu,
                                                        const float* __restrict__ su, int T, int max_active,
                                                        int route) {
  extern __shared__ __align__(16) int smi[];
  __shared__ float4 red[512];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
  const int npass = cdiv(T, MC);
  const int upe = D.inter / 8;
  const int per_slot = upe * npass;
  const int stride = gridDim.x;
  const ActCache A(smi, max_active, T * D.NS);
  uint4 va[MNB], vb[MNB];
  Q4Scales<MNB> qs;
  const WT *wlo = Wg, *whi = Wu;
  auto set_rows_e = [&](int e, int it) {
    const int r = ((it % per_slot) / npass) * 8 + g;
    wlo = stack_row(Wg, e, D.inter, r, D.h, &qs.lo);
    whi = stack_row(Wu, e, D.inter, r, D.h, &qs.hi);
  };
  const int it0 = blockIdx.x;
  const bool pre = it0 < D.S * per_slot;             // shared-expert item: expert known now
  if (pre) {
    set_rows_e(D.E + it0 / per_slot, it0);
    mma_load_batch<WT, MNB>(va, vb, wlo, whi, D.h, warp, qs);
  }
  pdl_wait();
  pdl_trigger();
  if (route) {
    float* lg = reinterpret_cast<float*>(smi + ActCache::words(max_active, T * D.NS));
    int* ids = reinterpret_cast<int*>(lg + T * D.E);
    float* wts = reinterpret_cast<float*>(ids + T * D.k);
    int* scratch = reinterpret_cast<int*>(wts + T * D.k);
    route_in_block(D, B, A, T, lg, ids, wts, scratch);
  } else {
    copy_active(B, A, max_active, T * D.NS);
  }
  const int nitems = *A.nact * per_slot;
  auto valid = [&](int it) { return ((it % per_slot) % npass) * MC < A.cnt[it / per_slot]; };
  auto next_valid = [&](int it) {
    while (it < nitems && !valid(it)) it += stride;
    return it;
  };
  int it = next_valid(it0);
  if (it < nitems && !(pre && it == it0)) {
    set_rows_e(A.ex[it / per_slot], it);
    mma_load_batch<WT, MNB>(va, vb, wlo, whi, D.h, warp, qs);
  }
  int par = 0;
  while (it < nitems) {
    const int slot = it / per_slot, rem = it % per_slot;
    const int j = (rem / npass) * 8 + g, p0 = (rem % npass) * MC;
    const int e = A.ex[slot];
    const int nvalid = min(MC, A.cnt[slot] - p0);
    const int* pairs = A.perm + A.off[slot] + p0;
    float c[4];
    mma_part<WT, MNB>(va, vb, wlo, whi, D.h, g < nvalid ? B.u + (size_t)(pairs[g] / D.NS) * D.h : nullptr, c, qs);
    const int nx = next_valid(it + stride);
    if (nx < nitems) {
      set_rows_e(A.ex[nx / per_slot], nx);
      mma_load_batch<WT, MNB>(va, vb, wlo, whi, D.h, warp, qs);
    }
    block_sum4(c, red, par);
    par ^= 1;
    if (warp == 0) {
      float s0 = 1.f, s1 = 1.f;
      if constexpr (IsQ4<WT>::v) {
        s0 = sg[e] * (1.0f / F16_OP_SCALE);
        s1 = su[e] * (1.0f / F16_OP_SCALE);
      } else {
        if (sg != nullptr) s0 = sg[(size_t)e * D.inter + j];
        if (su != nullptr) s1 = su[(size_t)e * D.inter + j];
      }
#pragma unroll
      for (int ee = 0; ee < 2; ++ee) {
        const int col = 2 * q + ee;
        if (col < nvalid) B.h_act[(size_t)pairs[col] * D.inter + j] = silu(c[ee] * s0) * (c[2 + ee] * s1);
      }
    }
    it = nx;
  }
}

// Expert down projection y[pair][o] = sum_j W_d[e][o][j] * h_act[pair][j].
template <class WT>
__global__ void __launch_bounds__(256, SBPS) k_down_m(Dims D, StepBuf B, const WT* __restrict__ Wd,
                                                      const float* __restrict__ sd, int T, int max_active) {
  extern __shared__ __align__(16) int smi[];
  __shared__ float4 red[512];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
  const int npass = cdiv(T, MC);
  const int upe = D.h / 16;
  const int per_slot = upe * npass;
  const int stride = gridDim.x;
  const ActCache A(smi, max_active, T * D.NS);
  uint4 va[MNB], vb[MNB];
  Q4Scales<MNB> qs;
  const WT *wlo = Wd, *whi = Wd;
  auto set_rows_e = [&](int e, int it) {
    const int o = ((it % per_slot) / npass) * 16 + g;
    wlo = stack_row(Wd, e, D.h, o, D.inter, &qs.lo);
    whi = stack_row(Wd, e, D.h, o + 8, D.inter, &qs.hi);
  };
  const int it0 = blockIdx.x;
  const bool pre = it0 < D.S * per_slot;
  if (pre) {
    set_rows_e(D.E + it0 / per_slot, it0);
    mma_load_batch<WT, MNB>(va, vb, wlo, whi, D.inter, warp, qs);
  }
  pdl_wait();
  pdl_trigger();
  copy_active(B, A, max_active, T * D.NS);
  const int nitems = *A.nact * per_slot;
  auto valid = [&](int it) { return ((it % per_slot) % npass) * MC < A.cnt[it / per_slot]; };
  auto next_valid = [&](int it) {
    while (it < nitems && !valid(it)) it += stride;
    return it;
  };
  int it = next_valid(it0);
  if (it < nitems && !(pre && it == it0)) {
    set_rows_e(A.ex[it / per_slot], it);
    mma_load_batch<WT, MNB>(va, vb, wlo, whi, D.inter, warp, qs);
  }
  int par = 0;
  while (it < nitems) {
    const int slot = it / per_slot, rem = it % per_slot;
    const int o = (rem / npass) * 16 + g, p0 = (rem % npass) * MC;
    const int e = A.ex[slot];
    const int nvalid = min(MC, A.cnt[slot] - p0);
    const int* pairs = A.perm + A.off[slot] + p0;
    float c[4];
    mma_part<WT, MNB>(va, vb, wlo, whi, D.inter, g < nvalid ? B.h_act + (size_t)pairs[g] * D.inter : nullptr, c,
                      qs);
    const int nx = next_valid(it + stride);
    if (nx < nitems) {
      set_rows_e(A.ex[nx / per_slot], nx);
      mma_load_batch<WT, MNB>(va, vb, wlo, whi, D.inter, warp, qs);
    }
    block_sum4(c, red, par);
    par ^= 1;
    if (warp == 0) {
      float s0 = 1.f, s1 = 1.f;
      if constexpr (IsQ4<WT>::v) s0 = s1 = sd[e] * (1.0f / F16_OP_SCALE);
      else if (sd != nullptr) { s0 = sd[(size_t)e * D.h + o]; s1 = sd[(size_t)e * D.h + o + 8]; }
#pragma unroll
      for (int ee = 0; ee < 2; ++ee) {
        const int col = 2 * q + ee;
        if (col >= nvalid) continue;
        float* y = B.y + (size_t)pairs[col] * D.h;
        y[o] = c[ee] * s0;
        y[o + 8] = c[2 + ee] * s1;
      }
    }
    it = nx;
  }
}

// ---------------------------------------------------------------------------
// Streamed expert GEMVs (steps of at most 8 columns, bf16 or e4m3 weights).
// The register form keeps one unit's weights in flight per block, so every
// unit costs a DRAM round trip; here a producer warp runs ahead over the
// block's units and copies each unit's rows by TMA into a ring of stages in
// shared memory (a stage: the unit's rows over KST of K, landing as
// [128-byte chunk][row][128 bytes], 128-byte swizzle), while the 8 consumer
// warps split each stage's K steps exactly as the register form splits a
// unit's (warp w: steps w, w + 8, ...; mma_step; block_sum4 in warp order),
// so a unit's arithmetic is the register form's. Units of the block's shared
// experts are issued before the kernel waits for the router. Every wait is
// bounded; a timed-out wait raises DERR_TIMEOUT and the kernel runs on to
// its end without touching the stage again (no barrier loses a member). Two
// blocks share an SM (2 x 152 blocks).
constexpr int FT_MAXSLOT = 8;

__device__ __forceinline__ void ft_tma3d(uint32_t dst, const CUtensorMap* map, int row, int chunk, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(row), "r"(chunk), "r"(bar)
      : "memory");
}

// 16 bytes of row r at byte offset kb of a stage box of RB rows.
template <int RB>
__device__ __forceinline__ uint4 ft_lds(uint32_t box, int r, int kb) {
  const uint32_t a = box + (uint32_t)((((kb >> 7) * RB + r) << 7) + ((((kb & 127) >> 4) ^ (r & 7)) << 4));
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}

// DUAL = 1: gate/up + SwiGLU (ma = gate rows, mb = up rows; a unit is gate
// rows j..j+7 with up rows j..j+7); DUAL = 0: down (ma; rows o..o+15).
template <class WT, int DUAL>
__global__ void __launch_bounds__(288, 2) k_ffn_t(const __grid_constant__ CUtensorMap ma,
                                                  const __grid_constant__ CUtensorMap mb, Dims D, StepBuf B, int* err,
                                                  const float* __restrict__ sa, const float* __restrict__ sb, int T,
                                                  int max_active, int route, int KST, int nslot) {
  constexpr int SK = MmaStep<WT>::K, EPL = MmaStep<WT>::EPL, ESZ = (int)sizeof(WT);
  constexpr int RB = DUAL ? 8 : 16;                          // rows of one box
  extern __shared__ __align__(16) int smi[];
  __shared__ __align__(8) uint64_t full[FT_MAXSLOT], empty[FT_MAXSLOT];
  __shared__ float4 red[512];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
  const int K = DUAL ? D.h : D.inter, rows_e = DUAL ? D.inter : D.h;
  const int per_slot = rows_e / RB;
  const int nkc = K / KST;
  const int box_bytes = RB * KST * ESZ, slot_bytes = (DUAL ? 2 : 1) * box_bytes;
  const ActCache A(smi, max_active, T * D.NS);
  const int words = DUAL ? gateup_words(D, T, max_active, route != 0) : ActCache::words(max_active, T * D.NS);
  const uint32_t ring = ((uint32_t)__cvta_generic_to_shared(smi + words) + 1023u) & ~1023u;
  auto bar = [](uint64_t* b) { return (uint32_t)__cvta_generic_to_shared(b); };
  if (threadIdx.x == 0) {
    for (int s = 0; s < nslot; ++s) {
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar(full + s)));
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 8;" ::"r"(bar(empty + s)));
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  const int G = gridDim.x, b0 = blockIdx.x;
  // stage t of this block: unit i = t / nkc (item b0 + i G), K part kc = t % nkc, slot t % nslot
  auto issue = [&](int t, int e) {                           // producer lane 0; false: gave up
    const int s = t % nslot;
    if (t >= nslot && !mbar_wait_deadline(bar(empty + s), ((t / nslot) - 1) & 1, err)) return false;
    const int it = b0 + (t / nkc) * G, kc = t % nkc;
    const int row = e * rows_e + (it % per_slot) * RB;
    const int chunk = kc * (KST * ESZ / 128);
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar(full + s)),
                 "r"((uint32_t)slot_bytes) : "memory");
    ft_tma3d(ring + s * slot_bytes, &ma, row, chunk, bar(full + s));
    if (DUAL) ft_tma3d(ring + s * slot_bytes + box_bytes, &mb, row, chunk, bar(full + s));
    return true;
  };
  // a block's first units of shared experts: known before the router has run
  int npre = 0;
  if (warp == 8 && lane == 0) {
    for (int t = 0; t < nslot; ++t) {
      const int it = b0 + (t / nkc) * G;
      if (it >= D.S * per_slot) break;
      issue(t, D.E + it / per_slot);
      npre = t + 1;
    }
  }
  pdl_wait();
  pdl_trigger();
  if (DUAL && route) {
    float* lg = reinterpret_cast<float*>(smi + ActCache::words(max_active, T * D.NS));
    int* ids = reinterpret_cast<int*>(lg + T * D.E);
    float* wts = reinterpret_cast<float*>(ids + T * D.k);
    int* scratch = reinterpret_cast<int*>(wts + T * D.k);
    route_in_block(D, B, A, T, lg, ids, wts, scratch);
  } else {
    copy_active(B, A, max_active, T * D.NS);
  }
  const int nitems = *A.nact * per_slot;
  const int n_my = b0 < nitems ? (nitems - b0 + G - 1) / G : 0;
  const int total = n_my * nkc;

  if (warp == 8) {
    // ---- producer ----
    int t = npre;
    if (lane == 0) {
      for (; t < total; ++t)
        if (!issue(t, A.ex[(b0 + (t / nkc) * G) / per_slot])) {
          atomicOr(err, DERR_TIMEOUT);
          break;
        }
      // the block's shared memory outlives every copy: wait (bounded) for the last ones
      for (int u = max(0, t - nslot); u < t; ++u) mbar_wait_deadline(bar(full + u % nslot), (u / nslot) & 1, nullptr);
    }
    return;
  }

  // ---- consumers: warps 0..7 ----
  float cp[2][4];
  const float* x = nullptr;
  int par = 0;
  for (int t = 0; t < total; ++t) {
    const int s = t % nslot, kc = t % nkc;
    const int it = b0 + (t / nkc) * G, slot = it / per_slot;
    const int nvalid = min(MC, A.cnt[slot]);
    const int* pairs = A.perm + A.off[slot];
    if (kc == 0) {
#pragma unroll
      for (int part = 0; part < 2; ++part)
#pragma unroll
        for (int i = 0; i < 4; ++i) cp[part][i] = 0.f;
      x = g < nvalid ? (DUAL ? B.u + (size_t)(pairs[g] / D.NS) * D.h : B.h_act + (size_t)pairs[g] * D.inter) : nullptr;
    }
    const bool ok = mbar_wait_deadline(bar(full + s), (t / nslot) & 1, err);
    if (!ok && lane == 0) atomicOr(err, DERR_TIMEOUT);
    if (ok) {
      const uint32_t box = ring + s * slot_bytes;
      for (int st = warp; st < KST / SK; st += 8) {
        const int kl = st * SK + EPL * q;                    // element within the stage
        const uint4 va = ft_lds<RB>(box, g, kl * ESZ);
        const uint4 vb = DUAL ? ft_lds<RB>(box + box_bytes, g, kl * ESZ) : ft_lds<RB>(box, g + 8, kl * ESZ);
        mma_step<WT, 2>(va, vb, 0u, 0u, kc * KST + kl, x, cp);
      }
    }
    __syncwarp();
    if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar(empty + s)) : "memory");
    if (kc != nkc - 1) continue;
    float c[4];
    sum_parts<2>(cp, c);
    block_sum4_w8(c, red, par);
    par ^= 1;
    if (warp != 0) continue;
    const int e = A.ex[slot];
    if constexpr (DUAL) {
      const int j = (it % per_slot) * 8 + g;
      const float s0 = sa != nullptr ? sa[(size_t)e * D.inter + j] : 1.f;
      const float s1 = sb != nullptr ? sb[(size_t)e * D.inter + j] : 1.f;
#pragma unroll
      for (int ee = 0; ee < 2; ++ee) {
        const int col = 2 * q + ee;
        if (col < nvalid) B.h_act[(size_t)pairs[col] * D.inter + j] = silu(c[ee] * s0) * (c[2 + ee] * s1);
      }
    } else {
      const int o = (it % per_slot) * 16 + g;
      const float s0 = sa != nullptr ? sa[(size_t)e * D.h + o] : 1.f;
      const float s1 = sa != nullptr ? sa[(size_t)e * D.h + o + 8] : 1.f;
#pragma unroll
      for (int ee = 0; ee < 2; ++ee) {
        const int col = 2 * q + ee;
        if (col >= nvalid) continue;
        float* y = B.y + (size_t)pairs[col] * D.h;
        y[o] = c[ee] * s0;
        y[o + 8] = c[2 + ee] * s1;
      }
    }
  }
}

// Final RMSNorm + LM head + greedy argmax (+ accept/commit), bf16 weights.
// Warp 0's lanes keep the running best (value, index) of the block's rows for
// their two columns; the block's candidates go to scratch and the last block
// reduces them (larger value wins, equal values keep the lower index).
__global__ void __launch_bounds__(256, SBPS) k_lmhead_m(Dims D, DevState S, StepBuf B, const bf16_t* __restrict__ W,
                                                        const float* __restrict__ gamma, const float* x, int T,
                                                        float* __restrict__ logits_dbg, int commit, int n_seq,
                                                        int K) {
  extern __shared__ __align__(16) float sm[];
  __shared__ float4 red[512];
  __shared__ int s_last;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
  const int nunits = D.V / 16;
  const int npass = cdiv(T, MC);
  float* inv = sm;
  float* xs = sm + ((T + 3) & ~3);
  uint4 va[MNB], vb[MNB];
  Q4Scales<MNB> qs;                      // unused: the LM head is bf16
  const bf16_t *wlo = W, *whi = W;
  auto set_rows = [&](int u) {
    wlo = W + (size_t)(u * 16 + g) * D.h;
    whi = W + (size_t)(u * 16 + g + 8) * D.h;
  };
  if ((int)blockIdx.x < nunits) {
    set_rows(blockIdx.x);
    mma_load_batch<bf16_t, MNB>(va, vb, wlo, whi, D.h, warp, qs);
  }
  pdl_wait();
  pdl_trigger();
  row_inv_rms(x, T, D.h, D.eps, inv);
  __syncthreads();
  int par = 0;
  for (int pass = 0; pass < npass; ++pass) {
    const int t0 = pass * MC, nvalid = min(MC, T - t0);
    if (pass > 0) __syncthreads();
    stage_cols(xs, x, t0, nvalid, D.h, inv, gamma);
    __syncthreads();
    float best[2] = {-INFINITY, -INFINITY};
    int bidx[2] = {0x7fffffff, 0x7fffffff};
    for (int u = blockIdx.x; u < nunits; u += gridDim.x) {
      float c[4];
      mma_part<bf16_t, MNB>(va, vb, wlo, whi, D.h, g < nvalid ? xs + g * (D.h + 4) : nullptr, c, qs);
      const int un = u + (int)gridDim.x < nunits ? u + gridDim.x : (pass + 1 < npass ? (int)blockIdx.x : -1);
      if (un >= 0) {
        set_rows(un);
        mma_load_batch<bf16_t, MNB>(va, vb, wlo, whi, D.h, warp, qs);
      }
      block_sum4(c, red, par);
      par ^= 1;
      if (warp != 0) continue;
      const int r0 = u * 16 + g;
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int col = 2 * q + e;
        if (logits_dbg != nullptr && col < nvalid) {
          logits_dbg[(size_t)(t0 + col) * D.V + r0] = c[e];
          logits_dbg[(size_t)(t0 + col) * D.V + r0 + 8] = c[2 + e];
        }
        const float k0 = am_key(c[e]), k1 = am_key(c[2 + e]);       // rows in increasing order
        if (k0 > best[e] || (k0 == best[e] && r0 < bidx[e])) { best[e] = k0; bidx[e] = r0; }
        if (k1 > best[e] || (k1 == best[e] && r0 + 8 < bidx[e])) { best[e] = k1; bidx[e] = r0 + 8; }
      }
    }
    if (warp == 0) {
      // reduce over the eight row groups (lane bits 2..4) for each column
#pragma unroll
      for (int e = 0; e < 2; ++e) {
#pragma unroll
        for (int o = 4; o <= 16; o <<= 1) {
          const float ov = __shfl_xor_sync(0xffffffffu, best[e], o);
          const int oi = __shfl_xor_sync(0xffffffffu, bidx[e], o);
          if (ov > best[e] || (ov == best[e] && oi < bidx[e])) { best[e] = ov; bidx[e] = oi; }
        }
        const int col = 2 * q + e;
        if (g == 0 && col < nvalid) {
          B.am_val[(size_t)(t0 + col) * B.n_vblocks + blockIdx.x] = best[e];
          B.am_idx[(size_t)(t0 + col) * B.n_vblocks + blockIdx.x] = bidx[e];
        }
      }
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    s_last = (atomicAdd(B.cnt_lm, 1) == (int)gridDim.x - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const int nc = gridDim.x;
  for (int row = warp; row < T; row += GEMV_WARPS) {
    const size_t base = (size_t)row * B.n_vblocks;
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    for (int i = lane; i < nc; i += 32) {
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
    if (lane == 0) B.g[row] = bi;
  }
  if (threadIdx.x == 0) *B.cnt_lm = 0;
  if (!commit) return;
  __syncthreads();
  __threadfence();
  for (int sq = threadIdx.x; sq < n_seq; sq += blockDim.x) commit_seq(D, S, B, sq, K, B.g);
}

// ---------------------------------------------------------------------------
static int grid_for(const Dims& D, int items) {
  const int want = cdiv(items, GEMV_WARPS);
  const int cap = D.n_sm * SBPS;
  return want < 1 ? 1 : (want < cap ? want : cap);
}

static int max_active_of(const Dims& D, int T) {
  return (D.E > 0 ? (D.E < T * D.k ? D.E : T * D.k) : 0) + D.S;
}

// The tensor-core forms serve bf16 / e4m3 weights whose widths are whole
// steps (32 bf16 or 64 e4m3 elements) and whose row counts split into
// 16-row units; fp32 weights (and other shapes) keep the FMA forms.
static bool mma_form(const Dims& D) {
  if (D.wdtype == 0) return false;
  const int sk = D.wdtype == 1 ? 32 : D.wdtype == 2 ? 64 : 128;
  return D.h % sk == 0 && (D.Hq * D.d) % sk == 0 && D.inter % sk == 0 && D.h % 16 == 0 && D.inter % 8 == 0 &&
         (D.d / 2) % 8 == 0 && D.V % 16 == 0 && D.h % 4 == 0;
}
static size_t mma_stage_bytes(const Dims& D, int T) { return (size_t)(((T + 3) & ~3) + MC * (D.h + 4)) * sizeof(float); }
// persistent grid for block-level units
static int grid_blocks(const Dims& D, int units) {
  const int cap = D.n_sm * SBPS;
  return units < 1 ? 1 : (units < cap ? units : cap);
}

void launch_qkv(const Dims& D, const DevState& S, const StepBuf& B, const LayerW& W, int layer, int T,
                const float* x, cudaStream_t st) {
  if (mma_form(D)) {
    const dim3 g(grid_blocks(D, (D.Hq + 2 * D.Hkv) * (D.d / 16))), b(256);
    const size_t sm = mma_stage_bytes(D, T);
    if (D.wdtype == 1) launch_k(k_qkv_m<bf16_t>, g, b, sm, st, D, S, B, W.attn_norm, (const bf16_t*)W.w_qkv, (const float*)nullptr, layer, T, x);
    else if (D.wdtype == 3) launch_k(k_qkv_m<fp4_t>, g, b, sm, st, D, S, B, W.attn_norm, (const fp4_t*)W.w_qkv, W.s_qkv, layer, T, x);
    else launch_k(k_qkv_m<fp8_t>, g, b, sm, st, D, S, B, W.attn_norm, (const fp8_t*)W.w_qkv, W.s_qkv, layer, T, x);
    return;
  }
  const int units = (D.Hq + 2 * D.Hkv) * (D.d / 4);
  const dim3 g(grid_for(D, units)), b(256);
  const size_t sm = (size_t)StageLayout(T, D.h).total * sizeof(float);
  switch (D.wdtype) {
    case 0: launch_k(k_qkv_s<float>, g, b, sm, st, D, S, B, W.attn_norm, (const float*)W.w_qkv, (const float*)nullptr, layer, T, x); break;
    case 1: launch_k(k_qkv_s<bf16_t>, g, b, sm, st, D, S, B, W.attn_norm, (const bf16_t*)W.w_qkv, (const float*)nullptr, layer, T, x); break;
    default: launch_k(k_qkv_s<fp8_t>, g, b, sm, st, D, S, B, W.attn_norm, (const fp8_t*)W.w_qkv, W.s_qkv, layer, T, x);
  }
}

void launch_oproj(const Dims& D, const StepBuf& B, const LayerW& W, int T, float* xres, cudaStream_t st) {
  if (mma_form(D)) {
    const dim3 g(grid_blocks(D, (D.h / 16) * cdiv(T, MC))), b(256);
    if (D.wdtype == 1) launch_k(k_oproj_m<bf16_t>, g, b, 0, st, D, B, (const bf16_t*)W.w_o, (const float*)nullptr, T, xres);
    else if (D.wdtype == 3) launch_k(k_oproj_m<fp4_t>, g, b, 0, st, D, B, (const fp4_t*)W.w_o, W.s_o, T, xres);
    else launch_k(k_oproj_m<fp8_t>, g, b, 0, st, D, B, (const fp8_t*)W.w_o, W.s_o, T, xres);
    return;
  }
  const int items = (D.h / 4) * cdiv(T, GEMV_TP);
  const dim3 g(grid_for(D, items)), b(256);
  switch (D.wdtype) {
    case 0: launch_k(k_oproj_s<float>, g, b, 0, st, D, B, (const float*)W.w_o, (const float*)nullptr, T, xres); break;
    case 1: launch_k(k_oproj_s<bf16_t>, g, b, 0, st, D, B, (const bf16_t*)W.w_o, (const float*)nullptr, T, xres); break;
    default: launch_k(k_oproj_s<fp8_t>, g, b, 0, st, D, B, (const fp8_t*)W.w_o, W.s_o, T, xres);
  }
}

// Ring slots of the streamed form that fit next to `words` ints of shared
// memory, two blocks to an SM (at least 2; 0: the streamed form does not fit).
static int ffn_slots(size_t words, int slot_bytes) {
  const long avail = 100L * 1024 - (long)words * 4 - 1024;   // two blocks an SM   // + 8.3 KB static: below 227 KB
  const int n = (int)std::min<long>(FT_MAXSLOT, avail / slot_bytes);
  return n >= 2 ? n : 0;
}

void launch_gateup(const Dims& D, const StepBuf& B, const LayerW& W, int T, int* err, cudaStream_t st) {
  const int ma = max_active_of(D, T);
  const bool route = route_in_gateup(T);
  const size_t sm = (size_t)gateup_words(D, T, ma, route) * sizeof(int);
  const int rt = route ? 1 : 0;
  if (W.ffn_map != nullptr && mma_form(D) && T <= MC && (D.wdtype == 1 || D.wdtype == 2)) {
    const int esz = D.wdtype == 1 ? 2 : 1, slot_bytes = 2 * 8 * W.kst_gu * esz;
    const int ns = ffn_slots(gateup_words(D, T, ma, route), slot_bytes);
    if (ns > 0) {
      const size_t smt = sm + 1024 + (size_t)ns * slot_bytes;
      if (D.wdtype == 1)
        launch_k(k_ffn_t<bf16_t, 1>, dim3(2 * D.n_sm), dim3(288), smt, st, W.ffn_map[0], W.ffn_map[1], D, B, err,
                 (const float*)nullptr, (const float*)nullptr, T, ma, rt, W.kst_gu, ns);
      else
        launch_k(k_ffn_t<fp8_t, 1>, dim3(2 * D.n_sm), dim3(288), smt, st, W.ffn_map[0], W.ffn_map[1], D, B, err,
                 W.s_gate, W.s_up, T, ma, rt, W.kst_gu, ns);
      return;
    }
  }
  if (mma_form(D)) {
    const dim3 g(grid_blocks(D, ma * (D.inter / 8) * cdiv(T, MC))), b(256);
    if (D.wdtype == 1)
      launch_k(k_gateup_m<bf16_t>, g, b, sm, st, D, B, (const bf16_t*)W.w_gate, (const float*)nullptr,
               (const bf16_t*)W.w_up, (const float*)nullptr, T, ma, rt);
    else if (D.wdtype == 3)
      launch_k(k_gateup_m<fp4_t>, g, b, sm, st, D, B, (const fp4_t*)W.w_gate, W.s_gate, (const fp4_t*)W.w_up,
               W.s_up, T, ma, rt);
    else
      launch_k(k_gateup_m<fp8_t>, g, b, sm, st, D, B, (const fp8_t*)W.w_gate, W.s_gate, (const fp8_t*)W.w_up,
               W.s_up, T, ma, rt);
    return;
  }
  const int items = ma * (D.inter / 2) * cdiv(T, GEMV_TP);
  const dim3 g(grid_for(D, items)), b(256);
  switch (D.wdtype) {
    case 0: launch_k(k_gateup_s<float>, g, b, sm, st, D, B, (const float*)W.w_gate, (const float*)nullptr,
                     (const float*)W.w_up, (const float*)nullptr, T, ma, rt); break;
    case 1: launch_k(k_gateup_s<bf16_t>, g, b, sm, st, D, B, (const bf16_t*)W.w_gate, (const float*)nullptr,
                     (const bf16_t*)W.w_up, (const float*)nullptr, T, ma, rt); break;
    default: launch_k(k_gateup_s<fp8_t>, g, b, sm, st, D, B, (const fp8_t*)W.w_gate, W.s_gate, (const fp8_t*)W.w_up,
                      W.s_up, T, ma, rt);
  }
}

void launch_down(const Dims& D, const StepBuf& B, const LayerW& W, int T, int* err, cudaStream_t st) {
  const int ma = max_active_of(D, T);
  const size_t sm = (size_t)ActCache::words(ma, T * D.NS) * sizeof(int);
  if (W.ffn_map != nullptr && mma_form(D) && T <= MC && (D.wdtype == 1 || D.wdtype == 2)) {
    const int esz = D.wdtype == 1 ? 2 : 1, slot_bytes = 16 * W.kst_dn * esz;
    const int ns = ffn_slots(ActCache::words(ma, T * D.NS), slot_bytes);
    if (ns > 0) {
      const size_t smt = sm + 1024 + (size_t)ns * slot_bytes;
      if (D.wdtype == 1)
        launch_k(k_ffn_t<bf16_t, 0>, dim3(2 * D.n_sm), dim3(288), smt, st, W.ffn_map[2], W.ffn_map[2], D, B, err,
                 (const float*)nullptr, (const float*)nullptr, T, ma, 0, W.kst_dn, ns);
      else
        launch_k(k_ffn_t<fp8_t, 0>, dim3(2 * D.n_sm), dim3(288), smt, st, W.ffn_map[2], W.ffn_map[2], D, B, err,
                 W.s_down, (const float*)nullptr, T, ma, 0, W.kst_dn, ns);
      return;
    }
  }
  if (mma_form(D)) {
    const dim3 g(grid_blocks(D, (D.h / 16) * ma * cdiv(T, MC))), b(256);
    if (D.wdtype == 1) launch_k(k_down_m<bf16_t>, g, b, sm, st, D, B, (const bf16_t*)W.w_down, (const float*)nullptr, T, ma);
    else if (D.wdtype == 3) launch_k(k_down_m<fp4_t>, g, b, sm, st, D, B, (const fp4_t*)W.w_down, W.s_down, T, ma);
    else launch_k(k_down_m<fp8_t>, g, b, sm, st, D, B, (const fp8_t*)W.w_down, W.s_down, T, ma);
    return;
  }
  const int items = (D.h / 4) * ma * cdiv(T, GEMV_TP);
  const dim3 g(grid_for(D, items)), b(256);
  switch (D.wdtype) {
    case 0: launch_k(k_down_s<float>, g, b, sm, st, D, B, (const float*)W.w_down, (const float*)nullptr, T, ma); break;
    case 1: launch_k(k_down_s<bf16_t>, g, b, sm, st, D, B, (const bf16_t*)W.w_down, (const float*)nullptr, T, ma); break;
    default: launch_k(k_down_s<fp8_t>, g, b, sm, st, D, B, (const fp8_t*)W.w_down, W.s_down, T, ma);
  }
}

void launch_combine(const Dims& D, const StepBuf& B, float* x, int T, cudaStream_t st) {
  const int n4 = T * D.h / 4;                      // hidden is a multiple of 4 (checked at init)
  int blocks = cdiv(n4, 256);
  if (blocks > 8 * D.n_sm) blocks = 8 * D.n_sm;
  launch_k(k_combine, dim3(blocks), dim3(256), 0, st, D, B, x, T);
}

// K elements a stage of the streamed expert GEMVs covers: K split into equal
// parts of whole TMA chunks (128 bytes) with 16 rows of a part <= 48 KB; 0
// when no split fits.
int ffn_stage_k(int K, int esz) {
  const int step = 128 / esz;                      // a TMA chunk; a multiple of the MMA step
  for (int n = 1; n <= K / step; ++n)
    if (K % n == 0 && (K / n) % step == 0 && 16L * (K / n) * esz <= 48 * 1024) return K / n;
  return 0;
}

int lmhead_step_warps(const Dims& D) { return grid_for(D, D.V / 4) * GEMV_WARPS; }

void launch_lmhead_step(const Dims& D, const DevState& S, const StepBuf& B, const void* lm_head,
                        const float* final_norm, const float* x, int T, float* logits_dbg, bool commit,
                        int n_seq, int K, cudaStream_t st) {
  if (mma_form(D)) {
    const dim3 g(grid_blocks(D, D.V / 16)), b(256);
    launch_k(k_lmhead_m, g, b, mma_stage_bytes(D, T), st, D, S, B, (const bf16_t*)lm_head, final_norm, x, T,
             logits_dbg, (int)commit, n_seq, K);
    return;
  }
  const dim3 g(grid_for(D, D.V / 4)), b(256);
  const size_t sm = (size_t)StageLayout(T, D.h).total * sizeof(float);
  if (D.act_f32)
    launch_k(k_lmhead_s<float>, g, b, sm, st, D, S, B, (const float*)lm_head, final_norm, x, T, logits_dbg,
             (int)commit, n_seq, K);
  else
    launch_k(k_lmhead_s<bf16_t>, g, b, sm, st, D, S, B, (const bf16_t*)lm_head, final_norm, x, T, logits_dbg,
             (int)commit, n_seq, K);
}

cudaError_t configure_stream_kernels() {
  cudaError_t e = cudaSuccess, r;
#define ALLOW(k) if ((r = allow_dyn_smem(k)) != cudaSuccess) e = r
  ALLOW(k_qkv_s<float>); ALLOW(k_qkv_s<bf16_t>); ALLOW(k_qkv_s<fp8_t>);
  ALLOW(k_gateup_s<float>); ALLOW(k_gateup_s<bf16_t>); ALLOW(k_gateup_s<fp8_t>);
  ALLOW(k_down_s<float>); ALLOW(k_down_s<bf16_t>); ALLOW(k_down_s<fp8_t>);
  ALLOW(k_lmhead_s<float>); ALLOW(k_lmhead_s<bf16_t>);
  ALLOW(k_qkv_m<bf16_t>); ALLOW(k_qkv_m<fp8_t>); ALLOW(k_gateup_m<bf16_t>); ALLOW(k_gateup_m<fp8_t>);
  ALLOW(k_down_m<bf16_t>); ALLOW(k_down_m<fp8_t>); ALLOW(k_lmhead_m);
  ALLOW(k_qkv_m<fp4_t>); ALLOW(k_gateup_m<fp4_t>); ALLOW(k_down_m<fp4_t>);
  ALLOW((k_ffn_t<bf16_t, 1>)); ALLOW((k_ffn_t<bf16_t, 0>)); ALLOW((k_ffn_t<fp8_t, 1>)); ALLOW((k_ffn_t<fp8_t, 0>));
#undef ALLOW
  return e;
}

}  // namespace spec
