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
// chunk) goes to scratch; the last block of a (group, kv head) to finish
// merges them in chunk order.
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

template <int D_HEAD, class KT>
__global__ void __launch_bounds__(ATT_THREADS) k_attn_part(Dims D, DevState S, StepBuf B, int layer, int T,
                                                           int R, int RG, int CS) {
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
  pdl_wait();
  pdl_trigger();
  const int hk = blockIdx.y;
  const int gps = (R + RG - 1) / RG;
  const int s = blockIdx.z / gps, sub = blockIdx.z % gps;
  const int r0 = s * R + sub * RG;
  if (r0 >= T) return;                              // whole group past T: no block of it counts
  const int nr = min(RG, min(R - sub * RG, T - r0));
  const int seq = B.row_seq[r0];
  const int maxpos = B.row_pos[r0 + nr - 1];
  const int G = D.Hq / D.Hkv;
  const int npairs = nr * G;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float scale = 1.0f / sqrtf((float)D_HEAD);
  const size_t head_off = (((size_t)layer * 2) * D.Hkv + hk) * D.P * D_HEAD;   // K of (layer, hk)
  const size_t v_off = (size_t)D.Hkv * D.P * D_HEAD;                            // K -> V
  const KT* kv = reinterpret_cast<const KT*>(S.kv);
  float* qw = Qw + warp * D_HEAD;
  float* pw = Pw + warp * ATT_CHUNK;

  for (int c = blockIdx.x; c * ATT_CHUNK <= maxpos; c += CS) {
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
    cp_async_wait_all();
    __syncthreads();
    // ---- one warp per (row, q head) pair ----
    for (int p = warp; p < npairs; p += ATT_THREADS / 32) {
      const int row = r0 + p / G;
      const int hq = hk * G + p % G;
      const int pos = B.row_pos[row];
      if (pos < k0) continue;                        // chunk lies after this row
      const float* qg = B.q + ((size_t)row * D.Hq + hq) * D_HEAD;
      for (int i = lane; i < D_HEAD; i += 32) qw[i] = qg[i];
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
      if (lane == 0) {
        B.att_ml[pidx * 2] = m;
        B.att_ml[pidx * 2 + 1] = l;
      }
      __syncwarp();
    }
  }
  // ---- the last of the CS chunk-slot blocks of this (group, kv head) merges ----
  __syncthreads();
  int* ctr = B.cnt_att + (size_t)blockIdx.z * D.Hkv + hk;
  if (threadIdx.x == 0) {
    __threadfence();
    s_last = (atomicAdd(ctr, 1) == (int)gridDim.x - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  // M = max_c m_c, L = sum_c l_c e^(m_c - M), o = sum_c o_c e^(m_c - M) / L,
  // chunks in order; one warp per (row, q head) of the group
  for (int p = warp; p < npairs; p += ATT_THREADS / 32) {
    const int row = r0 + p / G;
    const int hq = hk * G + p % G;
    const int nc = B.row_pos[row] / ATT_CHUNK + 1;
    const size_t base = ((size_t)row * D.Hq + hq) * B.n_chunk_max;
    float M = -INFINITY;
    for (int c = lane; c < nc; c += 32) M = fmaxf(M, __ldcg(B.att_ml + (base + c) * 2));
    M = warp_max(M);
    float Ll = 0.f;
    for (int c = lane; c < nc; c += 32)
      Ll = fmaf(__ldcg(B.att_ml + (base + c) * 2 + 1), expf(__ldcg(B.att_ml + (base + c) * 2) - M), Ll);
    const float L = warp_sum(Ll);
    float* out = B.o + (size_t)row * D.Hq * D_HEAD + (size_t)hq * D_HEAD;
    if constexpr (D_HEAD == 128) {
      float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int c = 0; c < nc; ++c) {
        const float w = expf(__ldcg(B.att_ml + (base + c) * 2) - M);
        const float4 v = __ldcg(reinterpret_cast<const float4*>(B.att_o + (base + c) * D_HEAD) + lane);
        o.x = fmaf(v.x, w, o.x); o.y = fmaf(v.y, w, o.y); o.z = fmaf(v.z, w, o.z); o.w = fmaf(v.w, w, o.w);
      }
      const float4 r = make_float4(o.x / L, o.y / L, o.z / L, o.w / L);
      reinterpret_cast<float4*>(out)[lane] = r;
      if (B.o_bf16 != nullptr) {
        const size_t e = (size_t)row * D.Hq * D_HEAD + (size_t)hq * D_HEAD + 4 * lane;
        const float rv[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint16_t hi = f_to_bf16(rv[i]);
          B.o_bf16[e + i] = hi;
          B.o_lo[e + i] = f_to_bf16(rv[i] - bf16_to_f(hi));
        }
      }
    } else {
      float2 o = make_float2(0.f, 0.f);
      for (int c = 0; c < nc; ++c) {
        const float w = expf(__ldcg(B.att_ml + (base + c) * 2) - M);
        const float2 v = __ldcg(reinterpret_cast<const float2*>(B.att_o + (base + c) * D_HEAD) + lane);
        o.x = fmaf(v.x, w, o.x); o.y = fmaf(v.y, w, o.y);
      }
      const float2 r = make_float2(o.x / L, o.y / L);
      reinterpret_cast<float2*>(out)[lane] = r;
      if (B.o_bf16 != nullptr) {
        const size_t e = (size_t)row * D.Hq * D_HEAD + (size_t)hq * D_HEAD + 2 * lane;
        const float rv[2] = {r.x, r.y};
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const uint16_t hi = f_to_bf16(rv[i]);
          B.o_bf16[e + i] = hi;
          B.o_lo[e + i] = f_to_bf16(rv[i] - bf16_to_f(hi));
        }
      }
    }
  }
  if (threadIdx.x == 0) *ctr = 0;
}

cudaError_t configure_attn_kernels() {
  cudaError_t e = cudaSuccess, r;
#define ALLOW(k) if ((r = allow_dyn_smem(k)) != cudaSuccess) e = r
  ALLOW((k_attn_part<128, float>)); ALLOW((k_attn_part<128, bf16_t>));
  ALLOW((k_attn_part<64, float>)); ALLOW((k_attn_part<64, bf16_t>));
#undef ALLOW
  return e;
}

void launch_attn_part(const Dims& D, const DevState& S, const StepBuf& B, int layer, int T, int R,
                      cudaStream_t st) {
  const int RG = R < 32 ? R : 32;
  const int groups = ((T + R - 1) / R) * ((R + RG - 1) / RG);
  // chunk slots: enough blocks to fill the GPU when few groups are live
  int CS = (2 * D.n_sm + groups * D.Hkv - 1) / (groups * D.Hkv);
  if (CS < 1) CS = 1;
  if (CS > B.n_chunk_max) CS = B.n_chunk_max;
  const dim3 grid(CS, D.Hkv, groups), blk(ATT_THREADS);
  if (D.d == 128) {
    if (D.act_f32) launch_k(k_attn_part<128, float>, grid, blk, AttSmem<128, float>::total, st, D, S, B, layer, T, R, RG, CS);
    else launch_k(k_attn_part<128, bf16_t>, grid, blk, AttSmem<128, bf16_t>::total, st, D, S, B, layer, T, R, RG, CS);
  } else {
    if (D.act_f32) launch_k(k_attn_part<64, float>, grid, blk, AttSmem<64, float>::total, st, D, S, B, layer, T, R, RG, CS);
    else launch_k(k_attn_part<64, bf16_t>, grid, blk, AttSmem<64, bf16_t>::total, st, D, S, B, layer, T, R, RG, CS);
  }
}

}  // namespace spec
