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
#include "gemv.cuh"
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

// Work list: per-group chunk counts -> exclusive prefix s_pref[0..n_groups]
// (warp 0; lane l owns groups [l*per, (l+1)*per)), then a block barrier.
__device__ __forceinline__ void att_prefix(const StepBuf& B, int T, int R, int RG, int n_groups, int* s_pref) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
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
}

// The item's group: s_pref[g] <= q < s_pref[g + 1] (the last such g is never empty).
__device__ __forceinline__ int att_group_of(const int* s_pref, int n_groups, int q) {
  int lo = 0, hi = n_groups;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (s_pref[mid] <= q) lo = mid; else hi = mid;
  }
  return lo;
}

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
  att_prefix(B, T, R, RG, n_groups, s_pref);
  const int G = D.Hq / D.Hkv;
  const float scale = 1.0f / sqrtf((float)D_HEAD);
  const size_t v_off = (size_t)D.Hkv * D.P * D_HEAD;                            // K -> V
  const KT* kv = reinterpret_cast<const KT*>(S.kv);
  float* qw = Qw + warp * D_HEAD;
  float* pw = Pw + warp * ATT_CHUNK;
  const int n_items = s_pref[n_groups] * D.Hkv;

  for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
    const int q = item / D.Hkv, hk = item % D.Hkv;
    const int g = att_group_of(s_pref, n_groups, q), c = q - s_pref[g];
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

// ===========================================================================
// Tensor-core form (bf16 K/V): warp-level mma.sync m16n8k16 with the chunk's
// 64 keys as M and the group's (row, q head) pairs as N (8 per tile, at most
// 32 per group: a group holds 32 / G rows). Per item:
//   S^T = K Q^T   (A = K rows by ldmatrix, B = Q as bf16 hi + lo: two MMAs),
//   softmax of each pair column over the chunk (fp32, causal mask),
//   O^T = V^T P^T (A = V by ldmatrix.trans, B = P as bf16 hi + lo).
// K and V are bf16 already, so the products are exact and the hi/lo split
// keeps Q and P near fp32. Warp w scores keys 16w..16w+15 and then outputs
// dims [D/4 w, D/4 (w+1)). Each pair column only meets its own Q and P, so a
// row's result does not depend on the group, the batch or its place in them.
constexpr int ATQ = 32;          // pairs per group at most (4 N tiles)

template <int D_HEAD>
struct AttTcSmem {
  static constexpr int KST = D_HEAD + 8;               // padded bf16 rows (ldmatrix without bank conflicts)
  static constexpr int PST = ATT_CHUNK + 8;
  static constexpr size_t k = 0;
  static constexpr size_t v = k + (size_t)ATT_CHUNK * KST * 2;
  static constexpr size_t qh = v + (size_t)ATT_CHUNK * KST * 2;
  static constexpr size_t ql = qh + (size_t)ATQ * KST * 2;
  static constexpr size_t ph = ql + (size_t)ATQ * KST * 2;
  static constexpr size_t pl = ph + (size_t)ATQ * PST * 2;
  static constexpr size_t sf = pl + (size_t)ATQ * PST * 2;      // fp32 S [64 keys][ATQ + 1]
  static constexpr size_t pg = sf + (size_t)ATT_CHUNK * (ATQ + 1) * 4;
  static constexpr size_t total = pg + ATT_CHUNK * 4;
};

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void* p) {
  const unsigned a = (unsigned)__cvta_generic_to_shared(p);
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(a));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], const void* p) {
  const unsigned a = (unsigned)__cvta_generic_to_shared(p);
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(a));
}
__device__ __forceinline__ void ldsm_x2(uint32_t& r0, uint32_t& r1, const void* p) {
  const unsigned a = (unsigned)__cvta_generic_to_shared(p);
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(a));
}
__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

template <int D_HEAD>
__global__ void __launch_bounds__(ATT_THREADS) k_attn_tc(Dims D, DevState S, StepBuf B, int layer, int T, int R,
                                                         int RG, int n_groups, int inline_merge) {
  using L = AttTcSmem<D_HEAD>;
  constexpr int KST = L::KST, PST = L::PST;
  constexpr int PPR = D_HEAD * 2 / 16;                 // 16-byte pieces per K/V row
  constexpr int DMT = D_HEAD / 16 / 4;                 // output dim tiles per warp
  extern __shared__ __align__(16) unsigned char smraw[];
  bf16_t* Ks = reinterpret_cast<bf16_t*>(smraw + L::k);
  bf16_t* Vs = reinterpret_cast<bf16_t*>(smraw + L::v);
  uint16_t* Qh = reinterpret_cast<uint16_t*>(smraw + L::qh);
  uint16_t* Ql = reinterpret_cast<uint16_t*>(smraw + L::ql);
  uint16_t* Ph = reinterpret_cast<uint16_t*>(smraw + L::ph);
  uint16_t* Pl = reinterpret_cast<uint16_t*>(smraw + L::pl);
  float* Sf = reinterpret_cast<float*>(smraw + L::sf);
  int* pg = reinterpret_cast<int*>(smraw + L::pg);
  __shared__ int s_last;
  __shared__ int s_pref[ATT_MAX_GROUPS + 1];
  pdl_wait();
  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, q4 = lane & 3;
  att_prefix(B, T, R, RG, n_groups, s_pref);
  const int G = D.Hq / D.Hkv;
  const float scale = 1.0f / sqrtf((float)D_HEAD);
  const size_t v_off = (size_t)D.Hkv * D.P * D_HEAD;
  const bf16_t* kv = reinterpret_cast<const bf16_t*>(S.kv);
  const int n_items = s_pref[n_groups] * D.Hkv;

  for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
    const int qi = item / D.Hkv, hk = item % D.Hkv;
    const int gi = att_group_of(s_pref, n_groups, qi), c = qi - s_pref[gi];
    const AttGroup grp(gi, T, R, RG);
    const int r0 = grp.r0, nr = grp.nr;
    const int seq = B.row_seq[r0];
    const int maxpos = B.row_pos[r0 + nr - 1];
    const int nch = maxpos / ATT_CHUNK + 1;
    const int npairs = nr * G;
    const int nnt = (npairs + 7) / 8;
    const int k0 = c * ATT_CHUNK;
    const int nk = min(ATT_CHUNK, maxpos + 1 - k0);
    const size_t head_off = (((size_t)layer * 2) * D.Hkv + hk) * D.P * D_HEAD;
    __syncthreads();
    // ---- pages, K/V pieces in flight, Q of the group's pairs as hi/lo ----
    for (int key = threadIdx.x; key < ATT_CHUNK; key += ATT_THREADS) {
      int page = -1;
      if (key < nk) {
        page = S.bt[(size_t)seq * D.max_pages + (k0 + key) / D.P];
        if (page < 0) atomicOr(S.err, DERR_PAGE);
      }
      pg[key] = page;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < 2 * ATT_CHUNK * PPR; i += ATT_THREADS) {
      const int isv = i >= ATT_CHUNK * PPR;
      const int j = isv ? i - ATT_CHUNK * PPR : i;
      const int key = j / PPR, piece = j % PPR;
      bf16_t* dst = (isv ? Vs : Ks) + key * KST + piece * 8;
      const int page = pg[key];
      if (page < 0) {                                 // keys past the chunk's end (or a missing page): zeros
        *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
        continue;
      }
      const size_t e = (size_t)page * D.page_elems + head_off + (isv ? v_off : 0) +
                       (size_t)((k0 + key) % D.P) * D_HEAD + piece * 8;
      cp_async16(dst, kv + e);
    }
    for (int i = threadIdx.x; i < nnt * 8 * (D_HEAD / 4); i += ATT_THREADS) {
      const int p = i / (D_HEAD / 4), d4 = (i % (D_HEAD / 4)) * 4;
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (p < npairs) {
        const int row = r0 + p / G, hq = hk * G + p % G;
        v = *reinterpret_cast<const float4*>(B.q + ((size_t)row * D.Hq + hq) * D_HEAD + d4);
      }
      uint32_t h0, l0, h1, l1;
      split_bf16x2(v.x, v.y, h0, l0);
      split_bf16x2(v.z, v.w, h1, l1);
      *reinterpret_cast<uint2*>(Qh + p * KST + d4) = make_uint2(h0, h1);
      *reinterpret_cast<uint2*>(Ql + p * KST + d4) = make_uint2(l0, l1);
    }
    cp_async_wait_all();
    __syncthreads();
    // ---- S^T (keys 16 warp .. +15) x pairs, scaled and causally masked, into Sf ----
    for (int nt = 0; nt < nnt; ++nt) {
      float ch[4] = {0.f, 0.f, 0.f, 0.f}, cl[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int ks = 0; ks < D_HEAD / 16; ++ks) {
        uint32_t a[4], bh0, bh1, bl0, bl1;
        ldsm_x4(a, Ks + (16 * warp + (lane & 7) + 8 * ((lane >> 3) & 1)) * KST + 16 * ks + 8 * (lane >> 4));
        const int prow = 8 * nt + (lane & 7), pcol = 16 * ks + 8 * ((lane >> 3) & 1);
        ldsm_x2(bh0, bh1, Qh + prow * KST + pcol);
        ldsm_x2(bl0, bl1, Ql + prow * KST + pcol);
        mma_bf16(ch, a, bh0, bh1);
        mma_bf16(cl, a, bl0, bl1);
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int key = 16 * warp + g + 8 * (e >> 1), p = 8 * nt + 2 * q4 + (e & 1);
        float sv = -INFINITY;
        if (p < npairs && key < nk && k0 + key <= B.row_pos[r0 + p / G]) sv = (ch[e] + cl[e]) * scale;
        Sf[key * (ATQ + 1) + p] = sv;
      }
    }
    __syncthreads();
    // ---- softmax of each pair over the chunk: P (hi/lo) and the partial (max, sum) ----
    for (int p = warp; p < nnt * 8; p += ATT_THREADS / 32) {
      const float s0 = Sf[lane * (ATQ + 1) + p], s1 = Sf[(lane + 32) * (ATQ + 1) + p];
      const float m = warp_max(fmaxf(s0, s1));
      float e0 = 0.f, e1 = 0.f;
      if (m != -INFINITY) {
        e0 = expf(s0 - m);
        e1 = expf(s1 - m);
      }
      const float l = warp_sum(e0 + e1);
      const uint16_t h0 = f_to_bf16(e0), h1 = f_to_bf16(e1);
      Ph[p * PST + lane] = h0;
      Ph[p * PST + lane + 32] = h1;
      Pl[p * PST + lane] = f_to_bf16(e0 - bf16_to_f(h0));
      Pl[p * PST + lane + 32] = f_to_bf16(e1 - bf16_to_f(h1));
      if (lane == 0 && p < npairs && m != -INFINITY) {
        const int row = r0 + p / G, hq = hk * G + p % G;
        const size_t pidx = ((size_t)row * D.Hq + hq) * B.n_chunk_max + c;
        reinterpret_cast<float2*>(B.att_ml)[pidx] = make_float2(m, l);
      }
    }
    __syncthreads();
    // ---- O^T (dims of this warp) x pairs -> chunk partials ----
    for (int nt = 0; nt < nnt; ++nt) {
      float oh[DMT][4], ol[DMT][4];
#pragma unroll
      for (int mt = 0; mt < DMT; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) { oh[mt][e] = 0.f; ol[mt][e] = 0.f; }
#pragma unroll
      for (int ks = 0; ks < ATT_CHUNK / 16; ++ks) {
        uint32_t bh0, bh1, bl0, bl1;
        const int prow = 8 * nt + (lane & 7), pcol = 16 * ks + 8 * ((lane >> 3) & 1);
        ldsm_x2(bh0, bh1, Ph + prow * PST + pcol);
        ldsm_x2(bl0, bl1, Pl + prow * PST + pcol);
#pragma unroll
        for (int mt = 0; mt < DMT; ++mt) {
          const int dm = 16 * (DMT * warp + mt);
          uint32_t a[4];
          // A = V^T [dims dm..dm+15][keys 16 ks..]: matrices (dims 0-7 | 8-15) x (keys 0-7 | 8-15)
          ldsm_x4_t(a, Vs + (16 * ks + (lane & 7) + 8 * (lane >> 4)) * KST + dm + 8 * ((lane >> 3) & 1));
          mma_bf16(oh[mt], a, bh0, bh1);
          mma_bf16(ol[mt], a, bl0, bl1);
        }
      }
#pragma unroll
      for (int mt = 0; mt < DMT; ++mt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int dim = 16 * (DMT * warp + mt) + g + 8 * (e >> 1), p = 8 * nt + 2 * q4 + (e & 1);
          if (p >= npairs) continue;
          const int row = r0 + p / G, hq = hk * G + p % G;
          if (B.row_pos[row] < k0) continue;              // chunk lies after this row: no partial
          const size_t pidx = ((size_t)row * D.Hq + hq) * B.n_chunk_max + c;
          B.att_o[pidx * D_HEAD + dim] = oh[mt][e] + ol[mt][e];
        }
      }
    }
    // ---- the last chunk of this (group, kv head) to finish merges its pairs ----
    if (!inline_merge) continue;
    __syncthreads();
    int* ctr = B.cnt_att + (size_t)gi * D.Hkv + hk;
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
  ALLOW(k_attn_tc<128>); ALLOW(k_attn_tc<64>);
#undef ALLOW
  return e;
}

// Pairs per group above which the merge runs as its own kernel.
constexpr int ATT_INLINE_PAIRS = 16;

// bf16 K/V with head dim 64 or 128 take the tensor-core form when a
// sequence's rows bring at least 16 (row, q head) pairs per kv head (block
// drafts, GQA); with fewer, most of each 8-column tile would be padding and
// the FMA form is faster. The choice depends only on the model (R is fixed
// by max_draft), so greedy and speculative steps share it.
static bool att_tc(const Dims& D, int R) {
  return !D.act_f32 && (D.d == 128 || D.d == 64) && D.Hq / D.Hkv <= ATQ && R * (D.Hq / D.Hkv) >= 16;
}

// Rows per group: the tensor-core form takes at most 32 (row, q head) pairs.
static int att_rg(const Dims& D, int R) {
  const int cap = att_tc(D, R) ? ATQ / (D.Hq / D.Hkv) : 32;
  return R < cap ? R : cap;
}

bool attn_separate_merge(const Dims& D, int R) { return att_rg(D, R) * (D.Hq / D.Hkv) > ATT_INLINE_PAIRS; }

int attn_groups(const Dims& D, int T, int R) {
  const int RG = att_rg(D, R);
  return ((T + R - 1) / R) * ((R + RG - 1) / RG);
}

void launch_attn_part(const Dims& D, const DevState& S, const StepBuf& B, int layer, int T, int R,
                      cudaStream_t st) {
  const int RG = att_rg(D, R);
  const int groups = attn_groups(D, T, R);
  const bool sep = attn_separate_merge(D, R);
  // fixed grid over the step's (group, chunk, kv head) items
  long long items = (long long)groups * B.n_chunk_max * D.Hkv;
  int blocks = 8 * D.n_sm;
  if (items < blocks) blocks = (int)items;
  const dim3 grid(blocks), blk(ATT_THREADS);
  const int im = sep ? 0 : 1;
  if (att_tc(D, R)) {
    if (D.d == 128) launch_k(k_attn_tc<128>, grid, blk, AttTcSmem<128>::total, st, D, S, B, layer, T, R, RG, groups, im);
    else launch_k(k_attn_tc<64>, grid, blk, AttTcSmem<64>::total, st, D, S, B, layer, T, R, RG, groups, im);
  } else if (D.d == 128) {
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
