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

template <int D_HEAD>
__global__ void __launch_bounds__(ATT_THREADS) k_attn_part(Dims D, DevState S, StepBuf B, int layer, int T,
                                                           int R, int RG, int CS) {
  constexpr int KLD = D_HEAD + 4;                  // padded row stride of K in shared memory
  extern __shared__ __align__(16) float sm[];
  float* Ks = sm;                                   // [64][KLD]
  float* Vs = Ks + ATT_CHUNK * KLD;                 // [64][D_HEAD]
  float* Qw = Vs + ATT_CHUNK * D_HEAD;              // [warps][D_HEAD]
  float* Pw = Qw + (ATT_THREADS / 32) * D_HEAD;     // [warps][64]
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
  float* qw = Qw + warp * D_HEAD;
  float* pw = Pw + warp * ATT_CHUNK;

  for (int c = blockIdx.x; c * ATT_CHUNK <= maxpos; c += CS) {
    const int k0 = c * ATT_CHUNK;
    const int nk = min(ATT_CHUNK, maxpos + 1 - k0);
    __syncthreads();
    // ---- stage K and V of keys [k0, k0 + nk) (16-byte vectors) ----
    constexpr int VPK = D_HEAD / 4;                  // float4 per key row
    for (int i = threadIdx.x; i < ATT_CHUNK * VPK; i += ATT_THREADS) {
      const int key = i / VPK, c4 = (i % VPK) * 4;
      float4 kv = make_float4(0.f, 0.f, 0.f, 0.f), vv = kv;
      if (key < nk) {
        const int pos = k0 + key;
        const int page = S.bt[(size_t)seq * D.max_pages + pos / D.P];
        if (page >= 0) {
          const size_t e = (size_t)page * D.page_elems + head_off + (size_t)(pos % D.P) * D_HEAD + c4;
          if (D.act_f32) {
            const float* kvp = reinterpret_cast<const float*>(S.kv);
            kv = *reinterpret_cast<const float4*>(kvp + e);
            vv = *reinterpret_cast<const float4*>(kvp + e + v_off);
          } else {
            const uint16_t* kvp = reinterpret_cast<const uint16_t*>(S.kv);
            const uint2 a = *reinterpret_cast<const uint2*>(kvp + e);
            const uint2 b = *reinterpret_cast<const uint2*>(kvp + e + v_off);
            kv = make_float4(__uint_as_float(a.x << 16), __uint_as_float(a.x & 0xFFFF0000u),
                             __uint_as_float(a.y << 16), __uint_as_float(a.y & 0xFFFF0000u));
            vv = make_float4(__uint_as_float(b.x << 16), __uint_as_float(b.x & 0xFFFF0000u),
                             __uint_as_float(b.y << 16), __uint_as_float(b.y & 0xFFFF0000u));
          }
        } else if (threadIdx.x == 0) {
          atomicOr(S.err, DERR_PAGE);
        }
      }
      *reinterpret_cast<float4*>(Ks + key * KLD + c4) = kv;
      *reinterpret_cast<float4*>(Vs + key * D_HEAD + c4) = vv;
    }
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
      // scores of keys lane and lane + 32
      float sc[2];
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        const int key = lane + 32 * h2;
        float acc = 0.f;
        const float* kr = Ks + key * KLD;
#pragma unroll 8
        for (int j = 0; j < D_HEAD; j += 4) {
          const float4 q4 = *reinterpret_cast<const float4*>(qw + j);
          const float4 k4 = *reinterpret_cast<const float4*>(kr + j);
          acc = fmaf(q4.x, k4.x, acc); acc = fmaf(q4.y, k4.y, acc);
          acc = fmaf(q4.z, k4.z, acc); acc = fmaf(q4.w, k4.w, acc);
        }
        sc[h2] = (k0 + key <= pos && key < nk) ? acc * scale : -INFINITY;
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
      if constexpr (D_HEAD == 128) {
        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int key = 0; key < nk; ++key) {
          const float pk = pw[key];
          const float4 v4 = *reinterpret_cast<const float4*>(Vs + key * D_HEAD + 4 * lane);
          o.x = fmaf(pk, v4.x, o.x); o.y = fmaf(pk, v4.y, o.y);
          o.z = fmaf(pk, v4.z, o.z); o.w = fmaf(pk, v4.w, o.w);
        }
        *reinterpret_cast<float4*>(og + 4 * lane) = o;
      } else {
        float2 o = make_float2(0.f, 0.f);
        for (int key = 0; key < nk; ++key) {
          const float pk = pw[key];
          const float2 v2 = *reinterpret_cast<const float2*>(Vs + key * D_HEAD + 2 * lane);
          o.x = fmaf(pk, v2.x, o.x); o.y = fmaf(pk, v2.y, o.y);
        }
        *reinterpret_cast<float2*>(og + 2 * lane) = o;
      }
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
      reinterpret_cast<float4*>(out)[lane] = make_float4(o.x / L, o.y / L, o.z / L, o.w / L);
    } else {
      float2 o = make_float2(0.f, 0.f);
      for (int c = 0; c < nc; ++c) {
        const float w = expf(__ldcg(B.att_ml + (base + c) * 2) - M);
        const float2 v = __ldcg(reinterpret_cast<const float2*>(B.att_o + (base + c) * D_HEAD) + lane);
        o.x = fmaf(v.x, w, o.x); o.y = fmaf(v.y, w, o.y);
      }
      reinterpret_cast<float2*>(out)[lane] = make_float2(o.x / L, o.y / L);
    }
  }
  if (threadIdx.x == 0) *ctr = 0;
}

cudaError_t configure_attn_kernels() {
  cudaError_t e = allow_dyn_smem(k_attn_part<128>);
  cudaError_t f = allow_dyn_smem(k_attn_part<64>);
  return e != cudaSuccess ? e : f;
}

void launch_attn_part(const Dims& D, const DevState& S, const StepBuf& B, int layer, int T, int R,
                      cudaStream_t st) {
  const int RG = R < 32 ? R : 32;
  const int groups = ((T + R - 1) / R) * ((R + RG - 1) / RG);
  // chunk slots: enough blocks to fill the GPU when few groups are live
  int CS = (304 + groups * D.Hkv - 1) / (groups * D.Hkv);
  if (CS < 1) CS = 1;
  if (CS > B.n_chunk_max) CS = B.n_chunk_max;
  dim3 grid(CS, D.Hkv, groups);
  const int dh = D.d;
  const size_t sm = (size_t)(ATT_CHUNK * (dh + 4) + ATT_CHUNK * dh + (ATT_THREADS / 32) * (dh + ATT_CHUNK)) *
                    sizeof(float);
  if (dh == 128) launch_k(k_attn_part<128>, grid, dim3(ATT_THREADS), sm, st, D, S, B, layer, T, R, RG, CS);
  else launch_k(k_attn_part<64>, grid, dim3(ATT_THREADS), sm, st, D, S, B, layer, T, R, RG, CS);
}


}  // namespace spec
