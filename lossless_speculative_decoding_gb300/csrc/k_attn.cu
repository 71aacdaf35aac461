// Verify attention over the paged KV cache, split over fixed 64-key chunks.
//
// Each verify row (the last committed token and the K drafts of a sequence,
// at consecutive positions n..n+K) attends causally to keys 0..pos. The keys
// are cut into chunks at absolute positions c*64 -- never at boundaries that
// depend on the number of rows, the batch or the page size -- so a row's
// result is the same whether it is scored alone (greedy step), with drafts,
// or during prefill. One block loads the K/V of one chunk of one kv head once
// (page by page, converted to fp32 in shared memory) and serves every query
// row of one sequence group and every q head that shares that kv head (GQA).
// A partial (unnormalised output, running max, running sum) per (row, head,
// chunk) goes to scratch and the partials are merged in chunk order: by the
// last block of a (group, kv head) to finish when a group has few (row, q
// head) pairs, else by a separate kernel with one warp per pair.
//
// Work list: the (group, chunk, kv head) items of the step are numbered
// group by group (each group has ceil((last position + 1) / 64) chunks) and a
// fixed grid strides over them, so long and short sequences share the GPU
// evenly and no block waits on a serial walk over a long context.
#include "common.cuh"
#include "kernels.h"

namespace spec {

constexpr int ATT_THREADS = 128;

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;" ::: "memory");
}

// Eight consecutive K elements of the storage type as floats.
template <class KT> __device__ __forceinline__ void load8(const KT* p, float* o);
template <> __device__ __forceinline__ void load8<float>(const float* p, float* o) {
  const float4 a = *reinterpret_cast<const float4*>(p), b = *reinterpret_cast<const float4*>(p + 4);
  o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w; o[4] = b.x; o[5] = b.y; o[6] = b.z; o[7] = b.w;
}
template <> __device__ __forceinline__ void load8<bf16_t>(const bf16_t* p, float* o) {
  const uint4 v = *reinterpret_cast<const uint4*>(p);
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    o[2 * i] = __uint_as_float(w[i] << 16);
    o[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}
// N (2 or 4) consecutive V elements of the storage type as floats.
template <class KT, int N> __device__ __forceinline__ void loadv(const KT* p, float* o);
template <> __device__ __forceinline__ void loadv<float, 4>(const float* p, float* o) {
  const float4 a = *reinterpret_cast<const float4*>(p);
  o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w;
}
template <> __device__ __forceinline__ void loadv<float, 2>(const float* p, float* o) {
  const float2 a = *reinterpret_cast<const float2*>(p);
  o[0] = a.x; o[1] = a.y;
}
template <> __device__ __forceinline__ void loadv<bf16_t, 4>(const bf16_t* p, float* o) {
  const uint2 v = *reinterpret_cast<const uint2*>(p);
  o[0] = __uint_as_float(v.x << 16); o[1] = __uint_as_float(v.x & 0xFFFF0000u);
  o[2] = __uint_as_float(v.y << 16); o[3] = __uint_as_float(v.y & 0xFFFF0000u);
}
template <> __device__ __forceinline__ void loadv<bf16_t, 2>(const bf16_t* p, float* o) {
  const uint32_t v = *reinterpret_cast<const uint32_t*>(p);
  o[0] = __uint_as_float(v << 16); o[1] = __uint_as_float(v & 0xFFFF0000u);
}

template <int D_HEAD, class KT>
struct AttSmem {
  static constexpr int KST = D_HEAD + 16 / (int)sizeof(KT);   // padded K row (one extra 16-byte piece)
  static constexpr size_t k_bytes = (size_t)ATT_CHUNK * KST * sizeof(KT);
  static constexpr size_t v_bytes = (size_t)ATT_CHUNK * D_HEAD * sizeof(KT);
  static constexpr size_t q_bytes = (size_t)(ATT_THREADS / 32) * D_HEAD * sizeof(float);
  static constexpr size_t p_bytes = (size_t)(ATT_THREADS / 32) * ATT_CHUNK * sizeof(float);
  static constexpr size_t total = k_bytes + v_bytes + q_bytes + p_bytes + ATT_CHUNK * sizeof(int);
};

// Merge the chunk partials of one (row, q head) pair, by one warp:
// M = max_c m_c, L = sum_c l_c e^(m_c - M), o = sum_c o_c e^(m_c - M) / L,
// chunks in order; writes o (fp32) and, when enabled, its hi/lo bf16 parts.
// Lanes fetch the (m, l) of 32 chunks at once and the output loop takes each
// chunk's weight from its lane, with eight chunks' partial rows in flight.
template <int D_HEAD>
__device__ __forceinline__ void merge_pair(const Dims& D, const StepBuf& B, int row, int hq) {
  const int lane = threadIdx.x & 31;
  const int nc = B.row_pos[row] / ATT_CHUNK + 1;
  const size_t base = ((size_t)row * D.Hq + hq) * B.n_chunk_max;
  const float2* ml = reinterpret_cast<const float2*>(B.att_ml) + base;
  float M = -INFINITY;
  for (int c = lane; c < nc; c += 32) M = fmaxf(M, __ldcg(ml + c).x);
  M = warp_max(M);
  constexpr int NV = D_HEAD / 32;
  float o[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i) o[i] = 0.f;
  float Ll = 0.f;
  for (int c0 = 0; c0 < nc; c0 += 32) {
    float w = 0.f;
    if (c0 + lane < nc) {
      const float2 v = __ldcg(ml + c0 + lane);
      w = expf(v.x - M);
      Ll = fmaf(v.y, w, Ll);
    }
    const int n = min(32, nc - c0);
    for (int j0 = 0; j0 < n; j0 += 8) {
      float vv[8][NV];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (j0 + u < n) {
          const float* v = B.att_o + (base + c0 + j0 + u) * D_HEAD + NV * lane;
          if constexpr (NV == 4) {
            const float4 t = __ldcg(reinterpret_cast<const float4*>(v));
            vv[u][0] = t.x; vv[u][1] = t.y; vv[u][2] = t.z; vv[u][3] = t.w;
          } else {
            const float2 t = __ldcg(reinterpret_cast<const float2*>(v));
            vv[u][0] = t.x; vv[u][1] = t.y;
          }
        }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const float wj = __shfl_sync(0xffffffffu, w, (j0 + u) & 31);
        if (j0 + u < n) {
#pragma unroll
          for (int i = 0; i < NV; ++i) o[i] = fmaf(vv[u][i], wj, o[i]);
        }
      }
    }
  }
  const float L = warp_sum(Ll);
  float* out = B.o + (size_t)row * D.Hq * D_HEAD + (size_t)hq * D_HEAD;
  float r[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i) r[i] = o[i] / L;
  if constexpr (NV == 4) reinterpret_cast<float4*>(out)[lane] = make_float4(r[0], r[1], r[2], r[3]);
  else reinterpret_cast<float2*>(out)[lane] = make_float2(r[0], r[1]);
  if (B.o_bf16 != nullptr) {
    const size_t e = (size_t)row * D.Hq * D_HEAD + (size_t)hq * D_HEAD + NV * lane;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const uint16_t hi = f_to_bf16(r[i]);
      B.o_bf16[e + i] = hi;
      B.o_lo[e + i] = f_to_bf16(r[i] - bf16_to_f(hi));
    }
  }
}

// Group g of the step: rows [r0, r0 + nr) of one sequence (nr = 0: past T).
struct AttGroup {
  int r0, nr;
  __device__ AttGroup(int g, int T, int R, int RG) {
    const int gps = (R + RG - 1) / RG;
    const int s = g / gps, sub = g % gps;
    r0 = s * R + sub * RG;
    nr = r0 < T ? min(RG, min(R - sub * RG, T - r0)) : 0;
  }
};

template <int D_HEAD, class KT>
__global__ void __launch_bounds__(ATT_THREADS) k_attn_part(Dims D, DevState S, StepBuf B, int layer, int T,
                                                           int R, int RG, int n_groups, int inline_merge) {
  using L = AttSmem<D_HEAD, KT>;
  constexpr int KST = L::KST;
  constexpr int PPR = D_HEAD * (int)sizeof(KT) / 16;          // 16-byte pieces per key row
  extern __shared__ __align__(16) unsigned char smraw[];
  KT* Ks = reinterpret_cast<KT*>(smraw);                        // [64][KST]
  KT* Vs = reinterpret_cast<KT*>(smraw + L::k_bytes);           // [64][D_HEAD]
  float* Qw = reinterpret_cast<float*>(smraw + L::k_bytes + L::v_bytes);    // [warps][D_HEAD]
  float* Pw = Qw + (ATT_THREADS / 32) * D_HEAD;                 // [warps][64]
  int* pg = reinterpret_cast<int*>(Pw + (ATT_THREADS / 32) * ATT_CHUNK);  // [64] page of each key
  __shared__ int s_last;
  __shared__ int s_pref[ATT_MAX_GROUPS + 1];          // chunk items before group g
  pdl_wait();
  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // ---- per-group chunk counts -> exclusive prefix (warp 0; lane l owns groups [l*per, (l+1)*per)) ----
  if (warp == 0) {
    const int per = (n_groups + 31) / 32, g0 = lane * per;
    int sum = 0;
    for (int i = 0; i < per; ++i) {
      const AttGroup a(g0 + i, T, R, RG);
      if (g0 + i < n_groups && a.nr > 0) sum += B.row_pos[a.r0 + a.nr - 1] / ATT_CHUNK + 1;
    }
    int inc = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += v;
    }
    int run = inc - sum;
    for (int i = 0; i < per; ++i) {
      if (g0 + i < n_groups) {
        s_pref[g0 + i] = run;
        const AttGroup a(g0 + i, T, R, RG);
        if (a.nr > 0) run += B.row_pos[a.r0 + a.nr - 1] / ATT_CHUNK + 1;
      }
    }
    if (lane == 31) s_pref[n_groups] = inc;
  }
  __syncthreads();
  const int G = D.Hq / D.Hkv;
  const float scale = 1.0f / sqrtf((float)D_HEAD);
  const size_t v_off = (size_t)D.Hkv * D.P * D_HEAD;                            // K -> V
  const KT* kv = reinterpret_cast<const KT*>(S.kv);
  float* qw = Qw + warp * D_HEAD;
  float* pw = Pw + warp * ATT_CHUNK;
  const int n_items = s_pref[n_groups] * D.Hkv;

  for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
    const int q = item / D.Hkv, hk = item % D.Hkv;
    int lo = 0, hi = n_groups;                        // group: s_pref[g] <= q < s_pref[g + 1]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s_pref[mid] <= q) lo = mid; else hi = mid;
    }
    const int g = lo, c = q - s_pref[g];
    const AttGroup grp(g, T, R, RG);
    const int r0 = grp.r0, nr = grp.nr;
    const int seq = B.row_seq[r0];
    const int maxpos = B.row_pos[r0 + nr - 1];
    const int nch = maxpos / ATT_CHUNK + 1;
    const int npairs = nr * G;
    const size_t head_off = (((size_t)layer * 2) * D.Hkv + hk) * D.P * D_HEAD;   // K of (layer, hk)
    {
      const int k0 = c * ATT_CHUNK;
      const int nk = min(ATT_CHUNK, maxpos + 1 - k0);
      __syncthreads();
      // ---- pages of the chunk's keys, then every 16-byte piece of K and V in flight at once ----
      for (int key = threadIdx.x; key < nk; key += ATT_THREADS) {
        const int page = S.bt[(size_t)seq * D.max_pages + (k0 + key) / D.P];
        pg[key] = page;
        if (page < 0) atomicOr(S.err, DERR_PAGE);
      }
      __syncthreads();
      for (int i = threadIdx.x; i < 2 * nk * PPR; i += ATT_THREADS) {
        const int isv = i >= nk * PPR;
        const int j = isv ? i - nk * PPR : i;
        const int key = j / PPR, piece = j % PPR;
        const int page = pg[key];
        if (page < 0) continue;
        const size_t e = (size_t)page * D.page_elems + head_off + (isv ? v_off : 0) +
                         (size_t)((k0 + key) % D.P) * D_HEAD + piece * (16 / sizeof(KT));
        KT* dst = isv ? Vs + key * D_HEAD + piece * (16 / sizeof(KT)) : Ks + key * KST + piece * (16 / sizeof(KT));
        cp_async16(dst, kv + e);
      }
      // the query of each warp's next pair is fetched into registers while
      // the K/V copies are in flight (and, later, while the current pair computes)
      constexpr int QPL = D_HEAD / 32;               // query elements per lane
      float qn[QPL];
      auto fetch_q = [&](int p) {
        if (p < npairs) {
          const float* qg = B.q + ((size_t)(r0 + p / G) * D.Hq + hk * G + p % G) * D_HEAD + QPL * lane;
#pragma unroll
          for (int i = 0; i < QPL; ++i) qn[i] = qg[i];
        }
      };
      fetch_q(warp);
      cp_async_wait_all();
      __syncthreads();
      // ---- one warp per (row, q head) pair ----
      for (int p = warp; p < npairs; p += ATT_THREADS / 32) {
        const int row = r0 + p / G;
        const int hq = hk * G + p % G;
        const int pos = B.row_pos[row];
#pragma unroll
        for (int i = 0; i < QPL; ++i) qw[QPL * lane + i] = qn[i];
        fetch_q(p + ATT_THREADS / 32);
        if (pos < k0) continue;                        // chunk lies after this row
        __syncwarp();
        // scores of keys lane and lane + 32 (padded K rows: conflict-free 16-byte reads)
        float sc[2];
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          const int key = lane + 32 * h2;
          float acc = 0.f;
          const KT* kr = Ks + key * KST;
#pragma unroll 4
          for (int j = 0; j < D_HEAD; j += 8) {
            float kf[8];
            load8<KT>(kr + j, kf);
            const float4 qa = *reinterpret_cast<const float4*>(qw + j);
            const float4 qb = *reinterpret_cast<const float4*>(qw + j + 4);
            acc = fmaf(qa.x, kf[0], acc); acc = fmaf(qa.y, kf[1], acc);
            acc = fmaf(qa.z, kf[2], acc); acc = fmaf(qa.w, kf[3], acc);
            acc = fmaf(qb.x, kf[4], acc); acc = fmaf(qb.y, kf[5], acc);
            acc = fmaf(qb.z, kf[6], acc); acc = fmaf(qb.w, kf[7], acc);
          }
          sc[h2] = (key < nk && k0 + key <= pos) ? acc * scale : -INFINITY;
        }
        const float m = warp_max(fmaxf(sc[0], sc[1]));
        const float p0 = expf(sc[0] - m), p1 = expf(sc[1] - m);
        const float l = warp_sum(p0 + p1);
        pw[lane] = p0;
        pw[lane + 32] = p1;
        __syncwarp();
        // o[j] = sum_key p[key] * V[key][j], keys in order
        const size_t pidx = ((size_t)row * D.Hq + hq) * B.n_chunk_max + c;
        float* og = B.att_o + pidx * D_HEAD;
        constexpr int NV = D_HEAD / 32;               // dims per lane (4 or 2)
        float o[NV];
#pragma unroll
        for (int i = 0; i < NV; ++i) o[i] = 0.f;
        for (int key = 0; key < nk; ++key) {
          const float pk = pw[key];
          float vf[NV];
          loadv<KT, NV>(Vs + key * D_HEAD + NV * lane, vf);
#pragma unroll
          for (int i = 0; i < NV; ++i) o[i] = fmaf(pk, vf[i], o[i]);
        }
        if constexpr (NV == 4) *reinterpret_cast<float4*>(og + 4 * lane) = make_float4(o[0], o[1], o[2], o[3]);
        else *reinterpret_cast<float2*>(og + 2 * lane) = make_float2(o[0], o[1]);
        if (lane == 0) reinterpret_cast<float2*>(B.att_ml)[pidx] = make_float2(m, l);
        __syncwarp();
      }
    }
    // ---- the last chunk of this (group, kv head) to finish merges its pairs ----
    if (!inline_merge) continue;
    __syncthreads();
    int* ctr = B.cnt_att + (size_t)g * D.Hkv + hk;
    if (threadIdx.x == 0) {
      __threadfence();
      s_last = (atomicAdd(ctr, 1) == nch - 1);
    }
    __syncthreads();
    if (!s_last) continue;
    __threadfence();
    for (int p = warp; p < npairs; p += ATT_THREADS / 32) merge_pair<D_HEAD>(D, B, r0 + p / G, hk * G + p % G);
    if (threadIdx.x == 0) *ctr = 0;
  }
}

// Standalone merge: one warp per (row, q head) pair of rows [0, T).
template <int D_HEAD>
__global__ void __launch_bounds__(256) k_attn_merge(Dims D, StepBuf B, int T) {
  pdl_wait();
  pdl_trigger();
  const int n = T * D.Hq;
  for (int p = blockIdx.x * 8 + (threadIdx.x >> 5); p < n; p += gridDim.x * 8) merge_pair<D_HEAD>(D, B, p / D.Hq, p % D.Hq);
}

cudaError_t configure_attn_kernels() {
  cudaError_t e = cudaSuccess, r;
#define ALLOW(k) if ((r = allow_dyn_smem(k)) != cudaSuccess) e = r
  ALLOW((k_attn_part<128, float>)); ALLOW((k_attn_part<128, bf16_t>));
  ALLOW((k_attn_part<64, float>)); ALLOW((k_attn_part<64, bf16_t>));
#undef ALLOW
  return e;
}

// Pairs per group above which the merge runs as its own kernel.
constexpr int ATT_INLINE_PAIRS = 16;

bool attn_separate_merge(const Dims& D, int R) {
  const int RG = R < 32 ? R : 32;
  return RG * (D.Hq / D.Hkv) > ATT_INLINE_PAIRS;
}

int attn_groups(int T, int R) {
  const int RG = R < 32 ? R : 32;
  return ((T + R - 1) / R) * ((R + RG - 1) / RG);
}

void launch_attn_part(const Dims& D, const DevState& S, const StepBuf& B, int layer, int T, int R,
                      cudaStream_t st) {
  const int RG = R < 32 ? R : 32;
  const int groups = attn_groups(T, R);
  const bool sep = attn_separate_merge(D, R);
  // fixed grid over the step's (group, chunk, kv head) items
  long long items = (long long)groups * B.n_chunk_max * D.Hkv;
  int blocks = 8 * D.n_sm;
  if (items < blocks) blocks = (int)items;
  const dim3 grid(blocks), blk(ATT_THREADS);
  const int im = sep ? 0 : 1;
  if (D.d == 128) {
    if (D.act_f32) launch_k(k_attn_part<128, float>, grid, blk, AttSmem<128, float>::total, st, D, S, B, layer, T, R, RG, groups, im);
    else launch_k(k_attn_part<128, bf16_t>, grid, blk, AttSmem<128, bf16_t>::total, st, D, S, B, layer, T, R, RG, groups, im);
  } else {
    if (D.act_f32) launch_k(k_attn_part<64, float>, grid, blk, AttSmem<64, float>::total, st, D, S, B, layer, T, R, RG, groups, im);
    else launch_k(k_attn_part<64, bf16_t>, grid, blk, AttSmem<64, bf16_t>::total, st, D, S, B, layer, T, R, RG, groups, im);
  }
  if (sep) {
    int mb = (T * D.Hq + 7) / 8;
    if (mb > 8 * D.n_sm) mb = 8 * D.n_sm;
    if (D.d == 128) launch_k(k_attn_merge<128>, dim3(mb), dim3(256), 0, st, D, B, T);
    else launch_k(k_attn_merge<64>, dim3(mb), dim3(256), 0, st, D, B, T);
  }
}

}  // namespace spec
