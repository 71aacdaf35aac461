// Verify attention over the paged KV cache, split over fixed 64-key chunks.
//
// Each verify row (the last committed token and the K drafts of a sequence,
// at consecutive positions n..n+K) attends causally to keys 0..pos. The keys
// are cut into chunks at absolute positions c*64 -- never at boundaries that
// depend on the number of rows, the batch or the page size -- so a row's
// result is the same whether it is scored alone (greedy step), with drafts,
// or during prefill. A chunk's K/V are read once per (row group, kv head) and
// serve every query row of the group and every q head sharing that kv head
// (GQA). A partial (unnormalised output, running max, running sum) per (row,
// head, chunk) goes to scratch and the partials are merged in chunk order: by
// the last chunk of a (group, kv head) to finish when the step has few such
// units and a group few pairs, else by a separate kernel with one warp per
// pair -- the same merge arithmetic either way.
//
// Two forms, chosen per model:
//  * bf16 K/V, head dim 64 or 128: k_attn_w, persistent blocks with a TMA
//    producer warp and mma.sync consumer warps (described below);
//  * fp32 K/V: k_attn_part, SIMT dot products per (row, q head) pair over a
//    chunk staged with cp.async, a fixed grid striding over the items, so
//    the fp32 model keeps exact fp32 arithmetic.
// Work list: the step's (group, chunk, kv head) items, numbered group by
// group from a per-block prefix over the groups' last positions (each group
// has ceil((last position + 1) / 64) chunks; the SIMT form takes a group's
// items chunk by chunk, the tensor-core form kv head by kv head), so long and
// short sequences share the GPU evenly and no block waits on a serial walk
// over a long context.
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
      uint16_t p[2];
      split_parts(r[i], D.op_f16, 2, p);
      B.o_bf16[e + i] = p[0];
      B.o_lo[e + i] = p[1];
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
// With s_maxpos / s_seq given, also records each group's last position and
// sequence.
__device__ __forceinline__ void att_prefix(const StepBuf& B, int T, int R, int RG, int n_groups, int* s_pref,
                                           int* s_maxpos = nullptr, int* s_seq = nullptr) {
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
        if (a.nr > 0) {
          const int mp = B.row_pos[a.r0 + a.nr - 1];
          run += mp / ATT_CHUNK + 1;
          if (s_maxpos) {
            s_maxpos[g0 + i] = mp;
            s_seq[g0 + i] = B.row_seq[a.r0];
          }
        }
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
  const size_t v_off = (size_t)D.P * D_HEAD;                                     // K -> V
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
    const size_t head_off = (((size_t)layer * D.Hkv + hk) * 2) * D.P * D_HEAD;   // K of (layer, hk)
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
// Tensor-core form (bf16 K/V): warp-level mma.sync m16n8k16. A consumer group
// of NW warps takes one (group, kv head, chunk) item at a time; its warp w
// owns the N tile of pairs 8w..8w+7 of the group (NW warps cover up to 8 NW
// (row, q head) pairs) and, per 64-key chunk:
//   S^T = K Q^T   (M = the 64 keys, A = K by ldmatrix, B = Q as bf16 hi + lo,
//                  both multiplied into the same accumulator),
//   softmax of each pair column over the chunk (fp32, causal mask; the
//                  column max and sum by shuffles inside the warp),
//   O^T = V^T P^T (M = head dims, A = V by ldmatrix.trans, B = P as bf16
//                  hi + lo through a small per-warp transpose buffer).
// K and V are bf16 already, so the products are exact and the hi/lo split
// keeps Q and P near fp32. Each pair column only meets its own Q and P, so a
// row's result does not depend on the group, the batch or its place in them.
//
// Streaming: items are ordered (group, kv head, chunk); every block takes one
// contiguous run of them, and its CG consumer groups take every CG-th item.
// One producer warp looks up the pages and issues the K/V of each item by TMA
// into a ring of NB chunk buffers (full / empty mbarriers, every wait
// bounded). The tensor map spans the paged pool (dims: 64 dims, key in page,
// 64-dim half, (layer, kv head, K|V) plane, page; box 64 dims x KB keys x all
// halves x K and V, 128-byte swizzle -- page sizes are multiples of 16 (of 64
// for KB = 64), so a box never straddles pages); boxes past the chunk's last
// key read page -1 (zero fill). Which block or group computes an item never
// changes its arithmetic.
constexpr int ATQ = 32;          // pairs per group at most (four warps)
constexpr int ATT_NB = 6;        // chunk buffers per block

template <int D_HEAD, int NW, int CG, int NB, int KB = 16>
struct AttWSmem {
  static constexpr int HB = ATT_CHUNK * 128;            // 64 dims of K or V for the chunk's keys
  static constexpr int BUF = 2 * (D_HEAD / 64) * HB;    // K and V of one chunk: ATT_CHUNK / KB boxes
  static constexpr int BOXB = BUF / (ATT_CHUNK / KB);   // one box: K then V of KB keys, all dims
  static constexpr int KPART = BOXB / 2;                // its K part
  static constexpr int PST = ATT_CHUNK + 8;             // P row stride (bf16), padded
  static constexpr int PW = 2 * 8 * PST * 2;            // one warp's P hi + lo [8 pairs][PST]
  static constexpr size_t total = 1024 + (size_t)NB * BUF + (size_t)CG * NW * PW;   // + alignment slack
};

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t a) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(a));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], uint32_t a) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(a));
}
__device__ __forceinline__ void ldsm_x2(uint32_t& r0, uint32_t& r1, uint32_t a) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(a));
}
__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// Barrier of one consumer group (named barrier 1 + cg, NW warps) that also
// reduces a flag: true when it holds in every thread of the group.
template <int NW>
__device__ __forceinline__ bool group_sync_and(int cg, bool v) {
  if constexpr (NW == 1) {
    return __all_sync(0xffffffffu, v);
  } else {
    uint32_t r;
    asm volatile("{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.and.pred q, %2, %3, p;\n selp.u32 %0, 1, 0, q;\n}\n"
                 : "=r"(r) : "r"((uint32_t)v), "r"(1 + cg), "r"(NW * 32) : "memory");
    return r != 0;
  }
}
template <int NW>
__device__ __forceinline__ void group_sync(int cg) {
  if constexpr (NW == 1) __syncwarp();
  else asm volatile("bar.sync %0, %1;" ::"r"(1 + cg), "r"(NW * 32) : "memory");
}
// 2^x by the hardware approximation (relative error about 2^-22); e^y is
// computed as 2^(y log2 e).
__device__ __forceinline__ float exp2_approx(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// Byte offset of 16-byte piece c (0..7) of row r in a 128-byte-swizzled tile.
__device__ __forceinline__ uint32_t sw128(int r, int c) { return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4)); }

// Shared address of dims col..col+7 of key `key` (0..63) of a chunk buffer,
// K (kv = 0) or V (kv = 1). The buffer holds the chunk's boxes of KB keys (16,
// or 64 when a page holds whole chunks) as the TMA writes them: box j = keys
// KB j .. KB j + KB - 1, its K part then its V part, each [64-dim half][key]
// rows of 128 bytes with the 128-byte swizzle (boxes and parts start on
// 1024-byte boundaries, so a row's swizzle is its index within the part).
// The rows of consecutive keys take consecutive swizzle phases, so an 8-key
// ldmatrix tile is conflict-free.
template <int HALVES, int KB>
__device__ __forceinline__ uint32_t kv_addr(uint32_t base, int key, int col, int kv) {
  constexpr int BOXB = KB * 2 * HALVES * 128, KPART = BOXB / 2;
  const int row = (col >> 6) * KB + key % KB;
  return base + (uint32_t)((key / KB) * BOXB + kv * KPART) + sw128(row, (col & 63) >> 3);
}

// Item i of the (group, kv head, chunk) order.
struct AttItem {
  int g, hk, c;
  __device__ AttItem(const int* s_pref, int n_groups, int Hkv, int i) {
    g = att_group_of(s_pref, n_groups, i / Hkv);     // s_pref[g] Hkv <= i
    const int nc = s_pref[g + 1] - s_pref[g], r = i - s_pref[g] * Hkv;
    hk = r / nc;
    c = r % nc;
  }
};

template <int D_HEAD, int NW, int CG, int NB, int KB>
__global__ void __launch_bounds__((CG * NW + 1) * 32, 1)
    k_attn_w(const __grid_constant__ CUtensorMap kvmap, Dims D, DevState S, StepBuf B, int layer, int T, int R,
             int RG, int n_groups, int inline_merge) {
  using L = AttWSmem<D_HEAD, NW, CG, NB, KB>;
  constexpr int NBOX = ATT_CHUNK / KB;                 // TMA boxes per chunk (4 or 1)
  constexpr int HALVES = D_HEAD / 64, HB = L::HB, BUF = L::BUF, PST = L::PST;
  constexpr int KS = D_HEAD / 16;                      // 16-wide K steps over the head dim
  constexpr int NCW = CG * NW;                         // consumer warps; the producer is warp NCW
  extern __shared__ unsigned char smraw[];
  const uint32_t bufs = ((uint32_t)__cvta_generic_to_shared(smraw) + 1023u) & ~1023u;   // NB x [K halves][V halves]
  __shared__ __align__(8) uint64_t full[NB], empty[NB];
  __shared__ int s_pref[ATT_MAX_GROUPS + 1], s_maxpos[ATT_MAX_GROUPS], s_seq[ATT_MAX_GROUPS];
  __shared__ int s_last[CG];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, q4 = lane & 3;
  auto bar_of = [&](uint64_t* b) { return (uint32_t)__cvta_generic_to_shared(b); };
  if (threadIdx.x == 0) {
    for (int b = 0; b < NB; ++b) {
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar_of(full + b)));
      asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar_of(empty + b)), "r"(NW));
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  pdl_wait();
  pdl_trigger();
  att_prefix(B, T, R, RG, n_groups, s_pref, s_maxpos, s_seq);   // ends with a block barrier
  const int n_items = s_pref[n_groups] * D.Hkv;
  const int per = (n_items + (int)gridDim.x - 1) / (int)gridDim.x;
  const int i0 = blockIdx.x * per, i1 = min(n_items, i0 + per);
  if (i0 >= i1) return;
  const int n = i1 - i0;

  if (warp == NCW) {
    // ---- producer: item k into buffer k % NB once its previous item is consumed ----
    // Items are resolved eight ahead, lane 4 u + j holding item kb + u's box j:
    // its page (-1 past the chunk's last key; a missing page sets the error
    // bit), the key of the box's first row and the item's (layer, kv head)
    // plane, so neither lookup latency nor the item arithmetic sits between a
    // freed buffer and its refill.
    struct Box { int page, key, plane; };
    auto lookup = [&](int kb) {
      const int kk = kb + (lane >> 2), j = lane & 3;
      Box x{-1, 0, 0};
      if (kk < n && j < NBOX) {
        const AttItem it(s_pref, n_groups, D.Hkv, i0 + kk);
        x.key = it.c * ATT_CHUNK + KB * j;
        x.plane = (layer * D.Hkv + it.hk) * 2;
        if (x.key <= s_maxpos[it.g]) {
          x.page = S.bt[(size_t)s_seq[it.g] * D.max_pages + x.key / D.P];
          if (x.page < 0) atomicOr(S.err, DERR_PAGE);
        }
      }
      return x;
    };
    Box pcur = lookup(0), pnext = lookup(8);
    int k = 0;
    for (; k < n; ++k) {
      const int b = k % NB;
      if (k > 0 && k % 8 == 0) {
        pcur = pnext;
        pnext = lookup(k + 8);
      }
      if (k >= NB && !mbar_wait_deadline(bar_of(empty + b), ((k / NB) - 1) & 1, S.err)) {
        if (lane == 0) atomicOr(S.err, DERR_TIMEOUT);
        break;
      }
      const int src = ((k % 8) << 2) | (lane & 3);
      const int page = __shfl_sync(0xffffffffu, pcur.page, src);
      const int key = __shfl_sync(0xffffffffu, pcur.key, src);
      const int plane = __shfl_sync(0xffffffffu, pcur.plane, src);
      if (lane == 0)
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar_of(full + b)), "r"((uint32_t)BUF)
                     : "memory");
      __syncwarp();
      if (lane < NBOX) {
        // lane j: the K and V (every dim) of keys key .. key + KB - 1, one box
        // of the (layer, kv head) plane pair
        const uint32_t dst = bufs + b * BUF + lane * L::BOXB;
        asm volatile(
            "cp.async.bulk.tensor.5d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5, %6}], [%7];"
            ::"r"(dst), "l"(reinterpret_cast<uint64_t>(&kvmap)), "r"(0), "r"(key % D.P), "r"(0), "r"(plane), "r"(page),
              "r"(bar_of(full + b))
            : "memory");
      }
    }
    // the block's shared memory outlives every copy: wait (bounded) for the
    // last phase issued into each buffer (already complete unless aborted)
    if (lane == 0)
      for (int q = max(0, k - NB); q < k; ++q) mbar_wait_deadline(bar_of(full + q % NB), (q / NB) & 1, nullptr);
    return;
  }

  // ---- consumer group cg, warp wl of it: pairs 8 wl .. 8 wl + 7 of the group ----
  const int cg = warp / NW, wl = warp % NW;
  const float scale = 1.0f / sqrtf((float)D_HEAD);
  const float scale_l2e = scale * 1.4426950408889634f;    // scale * log2(e)
  const int G = D.Hq / D.Hkv;
  const uint32_t ph = bufs + NB * BUF + warp * L::PW, pl = ph + 8 * PST * 2;
  int staged_g = -1, staged_hk = -1;
  uint32_t qh[KS][2], ql[KS][2];                       // B fragments of Q (this warp's pairs)
  int pos[2] = {-1, -1};                               // positions of this lane's two pair columns
  bool compact = false;                                // <= 4 pairs: hi parts in columns 0-3, lo in 4-7
  for (int k = cg; k < n; k += CG) {
    const int b = k % NB;
    const AttItem it(s_pref, n_groups, D.Hkv, i0 + k);
    const int gi = it.g, hk = it.hk, c = it.c;
    const AttGroup grp(gi, T, R, RG);
    const int r0 = grp.r0;
    const int maxpos = s_maxpos[gi];
    const int nch = maxpos / ATT_CHUNK + 1;
    const int npairs = grp.nr * G;
    const int k0 = c * ATT_CHUNK;
    const int nk = min(ATT_CHUNK, maxpos + 1 - k0);
    // ---- Q fragments and pair positions, when the (group, kv head) changes ----
    if (gi != staged_g || hk != staged_hk) {
      // compact form (at most 4 pairs, warp 0 only): column n < 4 is the hi
      // part of pair n, column n + 4 its lo part, so one MMA takes both and a
      // shuffle (lanes q4, q4 ^ 2) adds them; every column sum is the one the
      // two-MMA form computes, so a pair's bits do not depend on the form
      compact = npairs <= 4;
      const int p = compact ? (g & 3) : 8 * wl + g;
      const float* qr = nullptr;
      if (p < npairs) qr = B.q + ((size_t)(r0 + p / G) * D.Hq + hk * G + p % G) * D_HEAD;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          float2 v = make_float2(0.f, 0.f);
          if (qr) v = *reinterpret_cast<const float2*>(qr + 16 * ks + 2 * q4 + 8 * u);
          split_bf16x2(v.x, v.y, qh[ks][u], ql[ks][u]);
          if (compact && g >= 4) qh[ks][u] = ql[ks][u];
        }
      }
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int pj = compact ? 2 * (q4 & 1) + j : 8 * wl + 2 * q4 + j;
        pos[j] = pj < npairs ? B.row_pos[r0 + pj / G] : -1;
      }
      staged_g = gi;
      staged_hk = hk;
    }
    // ---- this item's chunk: wait, zero V rows past the last key, publish in the group ----
    const bool ok = mbar_wait_deadline(bar_of(full + b), (k / NB) & 1, S.err);
    const uint32_t kb = bufs + b * BUF;
    if (ok && nk < ATT_CHUNK) {
      for (int e = wl * 32 + lane; e < (ATT_CHUNK - nk) * HALVES * 8; e += NW * 32) {
        const int h = e / ((ATT_CHUNK - nk) * 8), r = nk + (e / 8) % (ATT_CHUNK - nk), pc = e % 8;
        const uint32_t za = kb + (uint32_t)((r / KB) * L::BOXB + L::KPART + (h * KB + r % KB) * 128 + pc * 16);
        asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(za), "r"(0u) : "memory");
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // before TMA refills this buffer
    }
    if (!group_sync_and<NW>(cg, ok)) {
      if (wl == 0 && lane == 0) atomicOr(S.err, DERR_TIMEOUT);
      break;
    }
    if (8 * wl < npairs) {
      // ---- S^T: four 16-key tiles x this warp's 8 pairs (hi and lo Q in
      // separate accumulators, added in that order) ----
      float sacc[4][4], slo[4][4];
#pragma unroll
      for (int mt = 0; mt < 4; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) sacc[mt][e] = slo[mt][e] = 0.f;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        const int col = 16 * ks + 8 * (lane >> 4);
        uint32_t a[4][4];                              // the K step's four key tiles, loaded before any MMA
#pragma unroll
        for (int mt = 0; mt < 4; ++mt)
          ldsm_x4(a[mt], kv_addr<HALVES, KB>(kb, 16 * mt + (lane & 7) + 8 * ((lane >> 3) & 1), col, 0));
#pragma unroll
        for (int mt = 0; mt < 4; ++mt) {
          mma_bf16(sacc[mt], a[mt], qh[ks][0], qh[ks][1]);
          if (!compact) mma_bf16(slo[mt], a[mt], ql[ks][0], ql[ks][1]);
        }
      }
#pragma unroll
      for (int mt = 0; mt < 4; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e)
          sacc[mt][e] += compact ? __shfl_xor_sync(0xffffffffu, sacc[mt][e], 2) : slo[mt][e];
      // ---- mask, column max / sum over the 64 keys: p = 2^((s - max) * scale * log2 e),
      // the chunk's max kept in scaled units (max(s * scale) = max(s) * scale) ----
      float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int mt = 0; mt < 4; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int key = 16 * mt + g + 8 * (e >> 1), j = e & 1;
          const float v = (key < nk && k0 + key <= pos[j]) ? sacc[mt][e] : -INFINITY;
          sacc[mt][e] = v;
          mx[j] = fmaxf(mx[j], v);
        }
      float sm[2] = {0.f, 0.f};
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) mx[j] = fmaxf(mx[j], __shfl_xor_sync(0xffffffffu, mx[j], o));
#pragma unroll
      for (int mt = 0; mt < 4; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int key = 16 * mt + g + 8 * (e >> 1), j = e & 1;
          const float pe = mx[j] == -INFINITY ? 0.f : exp2_approx((sacc[mt][e] - mx[j]) * scale_l2e);
          sm[j] += pe;
          const uint16_t hi = f_to_bf16(pe), lo = f_to_bf16(pe - bf16_to_f(hi));
          const uint32_t off = (uint32_t)(((2 * q4 + j) * PST + key) * 2);
          if (compact) {   // row 2 q4 + j: the hi part of a pair (q4 < 2) or the lo part (q4 >= 2)
            asm volatile("st.shared.u16 [%0], %1;" ::"r"(ph + off), "h"(q4 < 2 ? hi : lo) : "memory");
          } else {
            asm volatile("st.shared.u16 [%0], %1;" ::"r"(ph + off), "h"(hi) : "memory");
            asm volatile("st.shared.u16 [%0], %1;" ::"r"(pl + off), "h"(lo) : "memory");
          }
        }
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) sm[j] += __shfl_xor_sync(0xffffffffu, sm[j], o);
      if (g == 0 && (!compact || q4 < 2)) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int pj = compact ? 2 * q4 + j : 8 * wl + 2 * q4 + j;
          if (pj < npairs && mx[j] != -INFINITY) {
            const size_t pidx = ((size_t)(r0 + pj / G) * D.Hq + hk * G + pj % G) * B.n_chunk_max + c;
            reinterpret_cast<float2*>(B.att_ml)[pidx] = make_float2(mx[j] * scale, sm[j]);
          }
        }
      }
      __syncwarp();
      // ---- O^T: head dims x this warp's pairs, keys in 16-wide steps (the
      // hi and lo parts of P in separate accumulators, added in that order) ----
      float o[KS][4], olo[KS][4];
#pragma unroll
      for (int mt = 0; mt < KS; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[mt][e] = olo[mt][e] = 0.f;
#pragma unroll
      for (int ks = 0; ks < ATT_CHUNK / 16; ++ks) {
        uint32_t bh0, bh1, bl0 = 0, bl1 = 0;
        const uint32_t poff = (uint32_t)(((lane & 7) * PST + 16 * ks + 8 * ((lane >> 3) & 1)) * 2);
        ldsm_x2(bh0, bh1, ph + poff);
        if (!compact) ldsm_x2(bl0, bl1, pl + poff);
        const int key = 16 * ks + (lane & 7) + 8 * (lane >> 4);
        // one-warp groups load the key step's V tiles before any MMA (the
        // registers are there); wider groups interleave loads and MMAs
        constexpr int VB = NW == 1 ? KS : 1;
#pragma unroll
        for (int m0 = 0; m0 < KS; m0 += VB) {
          uint32_t a[VB][4];
#pragma unroll
          for (int mt = 0; mt < VB; ++mt)
            ldsm_x4_t(a[mt], kv_addr<HALVES, KB>(kb, key, 16 * (m0 + mt) + 8 * ((lane >> 3) & 1), 1));
#pragma unroll
          for (int mt = 0; mt < VB; ++mt) {
            mma_bf16(o[m0 + mt], a[mt], bh0, bh1);
            if (!compact) mma_bf16(olo[m0 + mt], a[mt], bl0, bl1);
          }
        }
      }
#pragma unroll
      for (int mt = 0; mt < KS; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[mt][e] += compact ? __shfl_xor_sync(0xffffffffu, o[mt][e], 2) : olo[mt][e];
      // the chunk's K/V are no longer read by this warp
      __syncwarp();
      if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar_of(empty + b)) : "memory");
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int pj = compact ? 2 * q4 + j : 8 * wl + 2 * q4 + j;
        if ((compact && q4 >= 2) || pj >= npairs || pos[j] < k0) continue;   // chunk after this row: no partial
        float* og = B.att_o + (((size_t)(r0 + pj / G) * D.Hq + hk * G + pj % G) * B.n_chunk_max + c) * D_HEAD;
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
          og[16 * mt + g] = o[mt][j];
          og[16 * mt + g + 8] = o[mt][2 + j];
        }
      }
    } else {
      __syncwarp();
      if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar_of(empty + b)) : "memory");
    }
    // ---- the last chunk of this (group, kv head) to finish merges its pairs ----
    if (!inline_merge) continue;
    __threadfence();
    group_sync<NW>(cg);
    int* ctr = B.cnt_att + (size_t)gi * D.Hkv + hk;
    if (wl == 0 && lane == 0) s_last[cg] = (atomicAdd(ctr, 1) == nch - 1);
    group_sync<NW>(cg);
    const bool last = s_last[cg] != 0;
    group_sync<NW>(cg);                                // s_last[cg] is rewritten for the group's next item
    if (!last) continue;
    __threadfence();
    for (int p = 8 * wl; p < min(npairs, 8 * wl + 8); ++p) merge_pair<D_HEAD>(D, B, r0 + p / G, hk * G + p % G);
    if (wl == 0 && lane == 0) *ctr = 0;
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
  ALLOW((k_attn_w<128, 1, 6, ATT_NB, 16>)); ALLOW((k_attn_w<128, 2, 2, ATT_NB, 16>)); ALLOW((k_attn_w<128, 4, 2, ATT_NB, 16>));
  ALLOW((k_attn_w<64, 1, 6, ATT_NB, 16>)); ALLOW((k_attn_w<64, 2, 2, ATT_NB, 16>)); ALLOW((k_attn_w<64, 4, 2, ATT_NB, 16>));
  ALLOW((k_attn_w<128, 1, 6, ATT_NB, 64>)); ALLOW((k_attn_w<128, 2, 2, ATT_NB, 64>)); ALLOW((k_attn_w<128, 4, 2, ATT_NB, 64>));
  ALLOW((k_attn_w<64, 1, 6, ATT_NB, 64>)); ALLOW((k_attn_w<64, 2, 2, ATT_NB, 64>)); ALLOW((k_attn_w<64, 4, 2, ATT_NB, 64>));
#undef ALLOW
  return e;
}

// Pairs per group above which the merge runs as its own kernel.
constexpr int ATT_INLINE_PAIRS = 16;
// (group, kv head) units of a step above which the merge runs as its own kernel.
constexpr int ATT_INLINE_UNITS = 64;

// bf16 K/V with head dim 64 or 128 take the tensor-core form (fp32 K/V the
// FMA form). The choice depends only on the model, so greedy and
// speculative steps share it.
static bool att_tc(const Dims& D, int R) {
  (void)R;
  return !D.act_f32 && (D.d == 128 || D.d == 64) && D.Hq / D.Hkv <= ATQ;
}

// Rows per group: the tensor-core form takes at most 32 (row, q head) pairs (four warps).
static int att_rg(const Dims& D, int R) {
  const int cap = att_tc(D, R) ? ATQ / (D.Hq / D.Hkv) : 32;
  return R < cap ? R : cap;
}

// The merge runs as its own kernel when a group has many pairs, or when the
// step has many (group, kv head) units (then per-chunk arrival counting
// costs more than a launch). Either way each pair is merged by the same
// merge_pair arithmetic, so the choice may depend on T.
bool attn_separate_merge(const Dims& D, int R, int T) {
  return att_rg(D, R) * (D.Hq / D.Hkv) > ATT_INLINE_PAIRS || attn_groups(D, T, R) * D.Hkv > ATT_INLINE_UNITS;
}

int attn_groups(const Dims& D, int T, int R) {
  const int RG = att_rg(D, R);
  return ((T + R - 1) / R) * ((R + RG - 1) / RG);
}

void launch_attn_part(const Dims& D, const DevState& S, const StepBuf& B, int layer, int T, int R,
                      const CUtensorMap& kvmap, cudaStream_t st) {
  const int RG = att_rg(D, R);
  const int groups = attn_groups(D, T, R);
  const bool sep = attn_separate_merge(D, R, T);
  const int im = sep ? 0 : 1;
  if (att_tc(D, R)) {
    // one persistent block per SM: a producer warp and consumer groups of
    // one warp per 8 pairs of a group
    const int nw = (RG * (D.Hq / D.Hkv) + 7) / 8;
#define ATT_W(DH, NW, CG)                                                                                     \
  if (att_box_keys(D) == 64)                                                                                  \
    launch_k(k_attn_w<DH, NW, CG, ATT_NB, 64>, dim3(D.n_sm), dim3((CG * NW + 1) * 32),                        \
             AttWSmem<DH, NW, CG, ATT_NB, 64>::total, st, kvmap, D, S, B, layer, T, R, RG, groups, im);       \
  else                                                                                                         \
    launch_k(k_attn_w<DH, NW, CG, ATT_NB, 16>, dim3(D.n_sm), dim3((CG * NW + 1) * 32),                        \
             AttWSmem<DH, NW, CG, ATT_NB, 16>::total, st, kvmap, D, S, B, layer, T, R, RG, groups, im)
    if (D.d == 128) {
      if (nw <= 1) { ATT_W(128, 1, 6); } else if (nw <= 2) { ATT_W(128, 2, 2); } else { ATT_W(128, 4, 2); }
    } else {
      if (nw <= 1) { ATT_W(64, 1, 6); } else if (nw <= 2) { ATT_W(64, 2, 2); } else { ATT_W(64, 4, 2); }
    }
#undef ATT_W
  } else {
    // fixed grid over the step's (group, chunk, kv head) items
    long long items = (long long)groups * B.n_chunk_max * D.Hkv;
    int blocks = 8 * D.n_sm;
    if (items < blocks) blocks = (int)items;
    const dim3 grid(blocks), blk(ATT_THREADS);
    if (D.d == 128) {
      if (D.act_f32) launch_k(k_attn_part<128, float>, grid, blk, AttSmem<128, float>::total, st, D, S, B, layer, T, R, RG, groups, im);
      else launch_k(k_attn_part<128, bf16_t>, grid, blk, AttSmem<128, bf16_t>::total, st, D, S, B, layer, T, R, RG, groups, im);
    } else {
      if (D.act_f32) launch_k(k_attn_part<64, float>, grid, blk, AttSmem<64, float>::total, st, D, S, B, layer, T, R, RG, groups, im);
      else launch_k(k_attn_part<64, bf16_t>, grid, blk, AttSmem<64, bf16_t>::total, st, D, S, B, layer, T, R, RG, groups, im);
    }
  }
  if (sep) {
    int mb = (T * D.Hq + 7) / 8;
    if (mb > 8 * D.n_sm) mb = 8 * D.n_sm;
    if (D.d == 128) launch_k(k_attn_merge<128>, dim3(mb), dim3(256), 0, st, D, B, T);
    else launch_k(k_attn_merge<64>, dim3(mb), dim3(256), 0, st, D, B, T);
  }
}

}  // namespace spec
