// Weight-streaming kernels of the verify step (persistent grids, PDL).
//
// At verify-step sizes every projection reads each weight once and uses it
// for only a few rows, so these kernels are bound by HBM bandwidth. Each
// kernel runs a persistent grid (two 256-thread blocks per SM); every warp
// walks work items (R = 4 weight rows x one pass of up to TP = 4 activation
// rows) with a grid stride, streaming weights with 16-byte non-allocating
// loads and reading activations through L1. Where the weights do not depend
// on the preceding kernel, the first chunk group is loaded before the
// programmatic-dependent-launch wait, so the fetch overlaps the predecessor's
// tail; the next item's first group is loaded before the current item's
// reduction.
//
// Fused epilogues: RMSNorm (per-row 1/rms computed once per block, gamma
// applied per column) for QKV and the LM head; RoPE + the paged KV write
// after QKV; the residual add after the output projection; SwiGLU after the
// expert gate/up projection; the in-order expert combine after the down
// projection (last warp per 4-column tile); the argmax (running per-warp
// best, last block reduces) and the accept/commit after the LM head.
// Every output's arithmetic is independent of T, of the batch and of the
// launch shape, which keeps speculative and greedy decoding bit-identical.
#include "gemv.cuh"
#include "kernels.h"

namespace spec {

constexpr int SG = 4;          // chunk groups in flight per lane
constexpr int SBPS = 2;        // persistent blocks per SM

__host__ __device__ static inline int cdiv(int a, int b) { return (a + b - 1) / b; }

// ---------------------------------------------------------------------------
// QKV projection + RoPE + paged KV write. Unit = rows {i0, i0+1, i0+d/2,
// i0+1+d/2} of one head (both halves of two rotary pairs in one warp).
template <class WT>
__global__ void __launch_bounds__(256, SBPS) k_qkv_s(Dims D, DevState S, StepBuf B, const float* __restrict__ gamma,
                                                     const WT* __restrict__ W, const float* __restrict__ scale,
                                                     int layer, int T) {
  extern __shared__ float inv[];                       // [T] 1/rms per row
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q4 = D.d / 4, half = D.d / 2;
  const int npass = cdiv(T, GEMV_TP);
  const int nitems = (D.Hq + 2 * D.Hkv) * q4 * npass;
  const int stride = gridDim.x * GEMV_WARPS;
  const int nch = D.h / Elt<WT>::per16;
  int it = blockIdx.x * GEMV_WARPS + warp;
  uint4 wv[SG][4];
  const WT* wr[4];
  auto set_rows = [&](int item) {
    const int unit = item / npass;
    const int base = (unit / q4) * D.d, i0 = 2 * (unit % q4);
    wr[0] = W + (size_t)(base + i0) * D.h;
    wr[1] = W + (size_t)(base + i0 + 1) * D.h;
    wr[2] = W + (size_t)(base + i0 + half) * D.h;
    wr[3] = W + (size_t)(base + i0 + 1 + half) * D.h;
  };
  if (it < nitems) {
    set_rows(it);
    load_group<WT, 4, SG>(wv, wr, nch, lane);
  }
  pdl_wait();
  pdl_trigger();
  row_inv_rms(B.x, T, D.h, D.eps, inv);
  __syncthreads();
  for (; it < nitems; it += stride) {
    const int unit = it / npass, pass = it % npass;
    const int head = unit / q4, i0 = 2 * (unit % q4), base = head * D.d;
    const int t0 = pass * GEMV_TP, nvalid = min(GEMV_TP, T - t0);
    const float* xr[GEMV_TP];
#pragma unroll
    for (int t = 0; t < GEMV_TP; ++t) xr[t] = t < nvalid ? B.x + (size_t)(t0 + t) * D.h : nullptr;
    float acc[16];
    unit_dot<WT, 4, GEMV_TP, SG>(wv, wr, D.h, xr, gamma, acc);
    if (it + stride < nitems) {
      set_rows(it + stride);
      load_group<WT, 4, SG>(wv, wr, nch, lane);
    }
    const float sum = reduce_scatter<16>(acc);
    const int v = (lane >> 1) & 15, r = v / GEMV_TP, t = v % GEMV_TP;
    const int rowW = base + i0 + (r & 1) + (r >= 2 ? half : 0);
    float val = sum * (t < nvalid ? inv[t0 + t] : 0.f);
    if (scale != nullptr) val *= scale[rowW];
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
      const float c = S.rope_cos[(size_t)pos * half + j], s = S.rope_sin[(size_t)pos * half + j];
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
                       ((((size_t)layer * 2 + is_v) * D.Hkv + hk) * D.P + (pos % D.P)) * D.d + dim;
    if (D.act_f32) reinterpret_cast<float*>(S.kv)[off] = outv;
    else reinterpret_cast<uint16_t*>(S.kv)[off] = f_to_bf16(outv);
  }
}

// ---------------------------------------------------------------------------
// Output projection + residual: x[t][o] += sum_k W_o[o][k] * attn[t][k].
template <class WT>
__global__ void __launch_bounds__(256, SBPS) k_oproj_s(Dims D, StepBuf B, const WT* __restrict__ W,
                                                       const float* __restrict__ scale, int T) {
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
    unit_dot<WT, 4, GEMV_TP, SG>(wv, wr, K, xr, nullptr, acc);
    if (it + stride < nitems) {
      set_rows(it + stride);
      load_group<WT, 4, SG>(wv, wr, nch, lane);
    }
    const float sum = reduce_scatter<16>(acc);
    const int v = (lane >> 1) & 15, r = v / GEMV_TP, t = v % GEMV_TP;
    if ((lane & 1) || t >= nvalid) continue;
    const int o = o0 + r;
    B.x[(size_t)(t0 + t) * D.h + o] += scale != nullptr ? sum * scale[o] : sum;
  }
}

// ---------------------------------------------------------------------------
// Expert gate/up + SwiGLU. Items: (active-expert slot, pair of output rows j,
// j+1, row pass); the unit streams gate rows j, j+1 and up rows j, j+1 and
// writes h_act[pair][j] = silu(gate) * up for the pass's routed pairs.
template <class WT>
__global__ void __launch_bounds__(256, SBPS) k_gateup_s(Dims D, StepBuf B, const WT* __restrict__ Wg,
                                                        const float* __restrict__ sg, const WT* __restrict__ Wu,
                                                        const float* __restrict__ su, int T, int max_active) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int npass = cdiv(T, GEMV_TP);
  const int upe = D.inter / 2;                          // units per expert
  const int per_slot = upe * npass;
  const int nch = D.h / Elt<WT>::per16;
  const int stride = gridDim.x * GEMV_WARPS;
  pdl_wait();
  pdl_trigger();
  const int n_active = *B.n_active;
  const int nitems = min(n_active, max_active) * per_slot;
  uint4 wv[SG][4];
  const WT* wr[4];
  for (int it = blockIdx.x * GEMV_WARPS + warp; it < nitems; it += stride) {
    const int slot = it / per_slot, rem = it % per_slot;
    const int j = (rem / npass) * 2, pass = rem % npass;
    const int cnt = B.act_cnt[slot];
    const int p0 = pass * GEMV_TP;
    if (p0 >= cnt) continue;
    const int e = B.act_expert[slot];
    const int nvalid = min(GEMV_TP, cnt - p0);
    const int* pairs = B.perm + B.act_off[slot] + p0;
    const size_t eb = (size_t)e * D.inter * D.h;
    wr[0] = Wg + eb + (size_t)j * D.h;
    wr[1] = Wg + eb + (size_t)(j + 1) * D.h;
    wr[2] = Wu + eb + (size_t)j * D.h;
    wr[3] = Wu + eb + (size_t)(j + 1) * D.h;
    load_group<WT, 4, SG>(wv, wr, nch, lane);
    int pr[GEMV_TP];
    const float* xr[GEMV_TP];
#pragma unroll
    for (int t = 0; t < GEMV_TP; ++t) {
      pr[t] = t < nvalid ? pairs[t] : 0;
      xr[t] = t < nvalid ? B.u + (size_t)(pr[t] / D.NS) * D.h : nullptr;
    }
    float acc[16];
    unit_dot<WT, 4, GEMV_TP, SG>(wv, wr, D.h, xr, nullptr, acc);
    const float sum = reduce_scatter<16>(acc);          // lane >> 1 = r*TP + t; r: gate j, gate j+1, up j, up j+1
    const float up = __shfl_sync(0xffffffffu, sum, (lane + 2 * 2 * GEMV_TP) & 31);
    const int v = (lane >> 1) & 15, r = v / GEMV_TP, t = v % GEMV_TP;
    if ((lane & 1) || r >= 2 || t >= nvalid) continue;
    const int jj = j + r;
    float g = sum, uu = up;
    if (sg != nullptr) { g *= sg[(size_t)e * D.inter + jj]; uu *= su[(size_t)e * D.inter + jj]; }
    B.h_act[(size_t)pr[t] * D.inter + jj] = silu(g) * uu;
  }
}

// ---------------------------------------------------------------------------
// Expert down projection y[pair][o] = sum_j W_d[e][o][j] * h_act[pair][j],
// then the combine: the last warp to finish a 4-column tile (over all active
// slots and passes) adds sum over slots s, in order, of w[r][s] * y[r*NS+s][o]
// (routed weight p, shared weight 1) to the residual x.
template <class WT>
__global__ void __launch_bounds__(256, SBPS) k_down_s(Dims D, StepBuf B, const WT* __restrict__ Wd,
                                                      const float* __restrict__ sd, int T, int max_active) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int npass = cdiv(T, GEMV_TP);
  const int tiles = D.h / 4;
  const int nch = D.inter / Elt<WT>::per16;
  const int stride = gridDim.x * GEMV_WARPS;
  pdl_wait();
  pdl_trigger();
  const int n_active = min(*B.n_active, max_active);
  // items are tile-major so the passes and slots of one tile are spread over warps
  const int per_tile = n_active * npass;
  const int nitems = tiles * per_tile;
  uint4 wv[SG][4];
  const WT* wr[4];
  for (int it = blockIdx.x * GEMV_WARPS + warp; it < nitems; it += stride) {
    const int tile = it / per_tile, rem = it % per_tile;
    const int slot = rem / npass, pass = rem % npass;
    const int cnt = B.act_cnt[slot];
    const int p0 = pass * GEMV_TP;
    if (p0 < cnt) {
      const int e = B.act_expert[slot];
      const int nvalid = min(GEMV_TP, cnt - p0);
      const int* pairs = B.perm + B.act_off[slot] + p0;
      const int o0 = tile * 4;
#pragma unroll
      for (int r = 0; r < 4; ++r) wr[r] = Wd + ((size_t)e * D.h + o0 + r) * D.inter;
      load_group<WT, 4, SG>(wv, wr, nch, lane);
      int pr[GEMV_TP];
      const float* xr[GEMV_TP];
#pragma unroll
      for (int t = 0; t < GEMV_TP; ++t) {
        pr[t] = t < nvalid ? pairs[t] : 0;
        xr[t] = t < nvalid ? B.h_act + (size_t)pr[t] * D.inter : nullptr;
      }
      float acc[16];
      unit_dot<WT, 4, GEMV_TP, SG>(wv, wr, D.inter, xr, nullptr, acc);
      const float sum = reduce_scatter<16>(acc);
      const int v = (lane >> 1) & 15, r = v / GEMV_TP, t = v % GEMV_TP;
      if (!(lane & 1) && t < nvalid) {
        const int o = o0 + r;
        B.y[(size_t)pr[t] * D.h + o] = sd != nullptr ? sum * sd[(size_t)e * D.h + o] : sum;
      }
    }
    // arrival of this item on its tile
    __threadfence();
    __syncwarp();
    int prev = 0;
    if (lane == 0) prev = atomicAdd(B.cnt_down + tile, 1);
    prev = __shfl_sync(0xffffffffu, prev, 0);
    if (prev != per_tile - 1) continue;
    __threadfence();
    for (int i = lane; i < T * 4; i += 32) {
      const int row = i >> 2, col = tile * 4 + (i & 3);
      float a = 0.f;
      for (int s2 = 0; s2 < D.NS; ++s2) {
        const float w = s2 < D.k ? B.wts[row * D.k + s2] : 1.f;
        a = fmaf(w, __ldcg(B.y + ((size_t)row * D.NS + s2) * D.h + col), a);
      }
      B.x[(size_t)row * D.h + col] += a;
    }
    if (lane == 0) B.cnt_down[tile] = 0;
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
                                                        const float* __restrict__ gamma, const float* __restrict__ x,
                                                        int T, float* __restrict__ logits_dbg, int commit, int n_seq,
                                                        int K) {
  extern __shared__ float inv[];                        // [T]
  __shared__ int s_last;
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
  row_inv_rms(x, T, D.h, D.eps, inv);
  __syncthreads();
  const int v = (lane >> 1) & 15, r = v / GEMV_TP, t = v % GEMV_TP;
  for (int pass = 0; pass < npass; ++pass) {
    const int t0 = pass * GEMV_TP, nvalid = min(GEMV_TP, T - t0);
    const float* xr[GEMV_TP];
#pragma unroll
    for (int tt = 0; tt < GEMV_TP; ++tt) xr[tt] = tt < nvalid ? x + (size_t)(t0 + tt) * D.h : nullptr;
    float best = -INFINITY;
    int bidx = 0x7fffffff;
    for (int u = gw; u < nunits; u += nw) {
      float acc[16];
      unit_dot<WT, 4, GEMV_TP, SG>(wv, wr, D.h, xr, gamma, acc);
      const int un = u + nw < nunits ? u + nw : (pass + 1 < npass ? gw : -1);
      if (un >= 0) {
        set_rows(un);
        load_group<WT, 4, SG>(wv, wr, nch, lane);
      }
      const float val = reduce_scatter<16>(acc) * (t < nvalid ? inv[t0 + t] : 0.f);
      const int vi = u * 4 + r;
      if (logits_dbg != nullptr && !(lane & 1) && t < nvalid) logits_dbg[(size_t)(t0 + t) * D.V + vi] = val;
      if (val > best) { best = val; bidx = vi; }
    }
    if (gw >= nunits && pass + 1 < npass) {
      // a warp without units still publishes an empty candidate below
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
    if (lane == 0) B.g[row] = bi;
  }
  if (threadIdx.x == 0) *B.cnt_lm = 0;
  if (!commit) return;
  __syncthreads();
  __threadfence();
  for (int s = threadIdx.x; s < n_seq; s += blockDim.x) commit_seq(D, S, B, s, K, B.g);
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

void launch_qkv(const Dims& D, const DevState& S, const StepBuf& B, const LayerW& W, int layer, int T,
                cudaStream_t st) {
  const int items = (D.Hq + 2 * D.Hkv) * (D.d / 4) * cdiv(T, GEMV_TP);
  const dim3 g(grid_for(D, items)), b(256);
  const size_t sm = (size_t)T * sizeof(float);
  switch (D.wdtype) {
    case 0: launch_k(k_qkv_s<float>, g, b, sm, st, D, S, B, W.attn_norm, (const float*)W.w_qkv, (const float*)nullptr, layer, T); break;
    case 1: launch_k(k_qkv_s<bf16_t>, g, b, sm, st, D, S, B, W.attn_norm, (const bf16_t*)W.w_qkv, (const float*)nullptr, layer, T); break;
    default: launch_k(k_qkv_s<fp8_t>, g, b, sm, st, D, S, B, W.attn_norm, (const fp8_t*)W.w_qkv, W.s_qkv, layer, T);
  }
}

void launch_oproj(const Dims& D, const StepBuf& B, const LayerW& W, int T, cudaStream_t st) {
  const int items = (D.h / 4) * cdiv(T, GEMV_TP);
  const dim3 g(grid_for(D, items)), b(256);
  switch (D.wdtype) {
    case 0: launch_k(k_oproj_s<float>, g, b, 0, st, D, B, (const float*)W.w_o, (const float*)nullptr, T); break;
    case 1: launch_k(k_oproj_s<bf16_t>, g, b, 0, st, D, B, (const bf16_t*)W.w_o, (const float*)nullptr, T); break;
    default: launch_k(k_oproj_s<fp8_t>, g, b, 0, st, D, B, (const fp8_t*)W.w_o, W.s_o, T);
  }
}

void launch_gateup(const Dims& D, const StepBuf& B, const LayerW& W, int T, cudaStream_t st) {
  const int ma = max_active_of(D, T);
  const int items = ma * (D.inter / 2) * cdiv(T, GEMV_TP);
  const dim3 g(grid_for(D, items)), b(256);
  switch (D.wdtype) {
    case 0: launch_k(k_gateup_s<float>, g, b, 0, st, D, B, (const float*)W.w_gate, (const float*)nullptr,
                     (const float*)W.w_up, (const float*)nullptr, T, ma); break;
    case 1: launch_k(k_gateup_s<bf16_t>, g, b, 0, st, D, B, (const bf16_t*)W.w_gate, (const float*)nullptr,
                     (const bf16_t*)W.w_up, (const float*)nullptr, T, ma); break;
    default: launch_k(k_gateup_s<fp8_t>, g, b, 0, st, D, B, (const fp8_t*)W.w_gate, W.s_gate, (const fp8_t*)W.w_up,
                      W.s_up, T, ma);
  }
}

void launch_down(const Dims& D, const StepBuf& B, const LayerW& W, int T, cudaStream_t st) {
  const int ma = max_active_of(D, T);
  const int items = (D.h / 4) * ma * cdiv(T, GEMV_TP);
  const dim3 g(grid_for(D, items)), b(256);
  switch (D.wdtype) {
    case 0: launch_k(k_down_s<float>, g, b, 0, st, D, B, (const float*)W.w_down, (const float*)nullptr, T, ma); break;
    case 1: launch_k(k_down_s<bf16_t>, g, b, 0, st, D, B, (const bf16_t*)W.w_down, (const float*)nullptr, T, ma); break;
    default: launch_k(k_down_s<fp8_t>, g, b, 0, st, D, B, (const fp8_t*)W.w_down, W.s_down, T, ma);
  }
}

int lmhead_step_warps(const Dims& D) { return grid_for(D, D.V / 4) * GEMV_WARPS; }

void launch_lmhead_step(const Dims& D, const DevState& S, const StepBuf& B, const void* lm_head,
                        const float* final_norm, const float* x, int T, float* logits_dbg, bool commit, int n_seq,
                        int K, cudaStream_t st) {
  const dim3 g(grid_for(D, D.V / 4)), b(256);
  const size_t sm = (size_t)T * sizeof(float);
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
  ALLOW(k_lmhead_s<float>); ALLOW(k_lmhead_s<bf16_t>);
#undef ALLOW
  return e;
}

}  // namespace spec
