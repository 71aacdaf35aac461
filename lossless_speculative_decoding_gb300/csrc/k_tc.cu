// Tensor-core (tcgen05) GEMM for verify steps and prefill at T >= 16 rows.
//
// D[m, n] = sum_k W[m, k] * X[n, k]: weights W (bf16, row-major = K-major)
// fill the MMA's M = 128 rows, activation rows X its N <= 128 columns, so a
// CTA streams one 128-row weight tile once for all of its tokens. The
// activations are given as two bf16 operands, X = X_hi + X_lo (about 16
// mantissa bits), and both are multiplied into the same fp32 accumulator, so
// the result keeps near-fp32 activation precision while the weights stay
// exact bf16. Tiles of 64 K-elements (one 128-byte swizzle row) are brought into
// shared memory by TMA (cp.async.bulk.tensor, 128-byte swizzle) through a
// multi-stage mbarrier pipeline; one thread issues tcgen05.mma into a TMEM
// accumulator (fp32, lane = weight row, column = token); four warps read it
// back with tcgen05.ld for the epilogue. Experts are groups: the activation
// rows of group g are rows [off_g, off_g + cnt_g) of a permuted buffer, and a
// CTA computes the columns of one group, so each token column only ever sees
// its own row of X -- its result does not depend on the other tokens.
//
// FP8 weights (e4m3, per-row fp32 scale applied in the epilogue): TMA brings
// the e4m3 tile unswizzled into a staging buffer, four converter warps widen
// it to bf16 -- exactly, every e4m3 value is a bf16 value -- into the
// 128-byte-swizzled operand tile and signal the MMA thread, so the tensor
// cores run the same bf16 MMA while HBM carries one byte per weight.
//
// Every wait on an mbarrier is bounded; a timeout sets an error bit, the CTA
// stops issuing work, frees its TMEM and returns.
#include <cuda_fp8.h>
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"

namespace spec {

constexpr int TC_BM = 128;            // weight rows per CTA (MMA M)
constexpr int TC_BK = 64;             // K elements per stage (128 bytes of bf16)
constexpr int TC_NSUB = 32;           // activation rows per TMA box
constexpr int TC_MAXN = 128;          // columns per CTA
constexpr uint32_t TC_WAIT_LIMIT = 1u << 20;
constexpr int TC_A_BYTES = TC_BM * TC_BK * 2;        // 16 KB
constexpr int TC_B_BYTES = TC_MAXN * TC_BK * 2;      // 16 KB (hi) + 16 KB (lo)
constexpr int TC_A8_BYTES = TC_BM * TC_BK;           // 8 KB e4m3 staging per weight operand

__host__ __device__ constexpr int tc_stages(int dual, int f8) { return f8 ? (dual ? 2 : 4) : (dual ? 3 : 4); }
__host__ __device__ constexpr int tc_stage_bytes(int dual, int f8) {
  return (TC_A_BYTES + (f8 ? TC_A8_BYTES : 0)) * (1 + dual) + 2 * TC_B_BYTES;
}
__host__ __device__ constexpr int tc_smem_bytes(int dual, int f8) {
  return tc_stages(dual, f8) * tc_stage_bytes(dual, f8) + 1024 + 256;
}
__host__ __device__ constexpr int tc_threads(int f8) { return f8 ? 256 : 128; }

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  for (uint32_t i = 0; i < TC_WAIT_LIMIT; ++i) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    if (ok) return true;
  }
  return false;
}

// Shared-memory matrix descriptor of a K-major bf16 tile stored as 128-byte
// rows with the 128-byte swizzle (8-row groups 1024 bytes apart).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);   // start address
  d |= (uint64_t)1 << 16;                      // leading byte offset (unused with this swizzle)
  d |= (uint64_t)(1024 >> 4) << 32;            // stride byte offset: 8 rows x 128 bytes
  d |= (uint64_t)1 << 46;                      // descriptor version
  d |= (uint64_t)2 << 61;                      // 128-byte swizzle
  return d;
}

// Instruction descriptor: bf16 x bf16 -> fp32, both operands K-major.
__device__ __forceinline__ uint32_t tc_idesc(int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(TC_BM >> 4) << 24);
}

__device__ __forceinline__ void tma_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar) : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Eight e4m3 values (one 8-byte word pair) as eight bf16 values.
__device__ __forceinline__ uint4 e4m3x8_to_bf16x8(uint2 v) {
  const uint32_t w[2] = {v.x, v.y};
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)((w[i] >> (16 * h)) & 0xFFFF), __NV_E4M3);
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hr));
      o[2 * i + h] = (__float_as_uint(f.x) >> 16) | (__float_as_uint(f.y) & 0xFFFF0000u);
    }
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// Stage s of the FP8 form: e4m3 staging [128 rows][64 B] -> bf16 tile [128
// rows][128 B] with the 128-byte swizzle (16-byte piece c of row r at
// (c ^ (r % 8)) * 16). 128 converter threads, 8 pieces each.
__device__ __forceinline__ void convert_tile(const unsigned char* stg, unsigned char* dst, int t) {
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int i = t + 128 * j, r = i >> 3, c = i & 7;
    const uint2 v = *reinterpret_cast<const uint2*>(stg + r * 64 + c * 8);
    *reinterpret_cast<uint4*>(dst + r * 128 + ((c ^ (r & 7)) << 4)) = e4m3x8_to_bf16x8(v);
  }
}

template <int DUAL, int F8>
__global__ void __launch_bounds__(tc_threads(F8), 1) k_tc_gemm(const __grid_constant__ CUtensorMap mapA,
                                                               const __grid_constant__ CUtensorMap mapA2,
                                                               const __grid_constant__ CUtensorMap mapB,
                                                               const __grid_constant__ CUtensorMap mapBlo, TcParams P) {
  constexpr int STAGES = tc_stages(DUAL, F8);
  constexpr int SB = tc_stage_bytes(DUAL, F8);
  // stage layout: [A bf16 (x2 if DUAL)][B hi][B lo][A e4m3 staging (x2 if DUAL), F8 only]
  constexpr int STG_OFF = TC_A_BYTES * (1 + DUAL) + 2 * TC_B_BYTES;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  // full[STAGES], empty[STAGES], done, conv[STAGES] (F8: converted tile ready)
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * SB);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 3 * STAGES + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- the CTA's group and columns (whole-CTA early exits happen before any set-up) ----
  const int mt = blockIdx.x, slot = blockIdx.y, nt = blockIdx.z;
  const int n_groups = P.g_n ? *P.g_n : (int)gridDim.y;
  if (slot >= n_groups) return;
  const int grp = P.g_expert ? P.g_expert[slot] : slot;
  const int off = P.g_off ? P.g_off[slot] : 0;
  const int cnt = P.g_cnt ? P.g_cnt[slot] : P.N;
  const int n0 = nt * TC_MAXN;
  if (n0 >= cnt) return;
  const int nrows = min(TC_MAXN, cnt - n0);
  const int nsub = (nrows + TC_NSUB - 1) / TC_NSUB;
  const int N = nsub * TC_NSUB;                       // MMA N: multiple of 32, <= 128
  const int KT = P.K / TC_BK;
  const int wrow = grp * P.Mg + mt * TC_BM;           // first weight row of the tile
  constexpr uint32_t NCOL = DUAL ? 2 * TC_MAXN : TC_MAXN;   // TMEM columns

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2 * STAGES + 1; ++i)
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(bars + i)));
    for (int i = 0; i < STAGES; ++i)    // one arrival per converter warp
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 4;" ::"r"(smem_u32(bars + 2 * STAGES + 1 + i)));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    *abort_flag = 0;
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(NCOL));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *tmem_slot;

  if (warp == 0 && lane == 0) {
    // ---- TMA producer ----
    const uint32_t bytes = (F8 ? TC_A8_BYTES : TC_A_BYTES) * (1 + DUAL) + (P.split ? 2 : 1) * nsub * TC_NSUB * TC_BK * 2;
    for (int kt = 0; kt < KT; ++kt) {
      const int s = kt % STAGES;
      if (kt >= STAGES && !mbar_wait(smem_u32(bars + STAGES + s), ((kt / STAGES) - 1) & 1)) {
        atomicOr(P.err, DERR_TIMEOUT);
        *abort_flag = 1;
        break;
      }
      unsigned char* st = smem + s * SB;
      const uint32_t full = smem_u32(bars + s);
      asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(full), "r"(bytes) : "memory");
      unsigned char* at = F8 ? st + STG_OFF : st;
      constexpr int AST = F8 ? TC_A8_BYTES : TC_A_BYTES;
      tma_2d(smem_u32(at), &mapA, kt * TC_BK, wrow, full);
      if (DUAL) tma_2d(smem_u32(at + AST), &mapA2, kt * TC_BK, wrow, full);
      unsigned char* bt = st + TC_A_BYTES * (1 + DUAL);
      for (int j = 0; j < nsub; ++j) {
        tma_2d(smem_u32(bt + j * TC_NSUB * TC_BK * 2), &mapB, kt * TC_BK, off + n0 + j * TC_NSUB, full);
        if (P.split)
          tma_2d(smem_u32(bt + TC_B_BYTES + j * TC_NSUB * TC_BK * 2), &mapBlo, kt * TC_BK, off + n0 + j * TC_NSUB,
                 full);
      }
    }
  } else if (warp == 1 && lane == 0) {
    // ---- MMA issuer ----
    const uint32_t idesc = tc_idesc(N);
    bool ok = true;
    for (int kt = 0; kt < KT && ok; ++kt) {
      const int s = kt % STAGES;
      // bf16: the TMA bytes of the stage; F8: the converters' signal (after those bytes)
      if (!mbar_wait(smem_u32(bars + (F8 ? 2 * STAGES + 1 : 0) + s), (kt / STAGES) & 1)) {
        atomicOr(P.err, DERR_TIMEOUT);
        *abort_flag = 1;
        ok = false;
        break;
      }
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const uint32_t a0 = smem_u32(smem + s * SB);
      const uint32_t b0 = a0 + TC_A_BYTES * (1 + DUAL);
#pragma unroll
      for (int k = 0; k < TC_BK / 16; ++k) {
        // hi then (optionally) lo activations into the same accumulator
        for (int part = 0; part < (P.split ? 2 : 1); ++part) {
          const uint64_t bd = sw128_desc(b0 + part * TC_B_BYTES + k * 32);
          const uint32_t acc = (kt | k | part) != 0;
          const uint64_t ad = sw128_desc(a0 + k * 32);
          asm volatile(
              "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
              " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n"
              ::"r"(tmem), "l"(ad), "l"(bd), "r"(idesc), "r"(acc));
          if (DUAL) {
            const uint64_t ad2 = sw128_desc(a0 + TC_A_BYTES + k * 32);
            asm volatile(
                "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
                " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n"
                ::"r"(tmem + (uint32_t)TC_MAXN), "l"(ad2), "l"(bd), "r"(idesc), "r"(acc));
          }
        }
      }
      asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                   ::"r"(smem_u32(bars + STAGES + s)) : "memory");
    }
    if (ok)
      asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                   ::"r"(smem_u32(bars + 2 * STAGES)) : "memory");
  } else if (F8 && warp >= 4) {
    // ---- converters: e4m3 staging -> swizzled bf16 operand tile ----
    const int t = threadIdx.x - 128;
    for (int kt = 0; kt < KT; ++kt) {
      const int s = kt % STAGES;
      if (!mbar_wait(smem_u32(bars + s), (kt / STAGES) & 1)) {
        if (lane == 0) atomicOr(P.err, DERR_TIMEOUT);
        break;
      }
      unsigned char* st = smem + s * SB;
      convert_tile(st + STG_OFF, st, t);
      if (DUAL) convert_tile(st + STG_OFF + TC_A8_BYTES, st + TC_A_BYTES, t);
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bars + 2 * STAGES + 1 + s)) : "memory");
    }
  }
  __syncwarp();

  // ---- epilogue: warp w holds TMEM lanes 32w..32w+31 = weight rows ----
  const bool have = __syncthreads_and(mbar_wait(smem_u32(bars + 2 * STAGES), 0)) != 0;   // block-uniform
  if (!have && threadIdx.x == 0) atomicOr(P.err, DERR_TIMEOUT);
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  if (warp < 4) {
  const int m = warp * 32 + lane;                     // row within the tile
  const int col = mt * TC_BM + m;                     // output feature (row within the group)
  const float sc = (P.scale && have) ? P.scale[wrow + m] : 1.f;
  const float sc2 = (DUAL && P.scale2 && have) ? P.scale2[wrow + m] : 1.f;
  const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
  __shared__ float red_v[4][TC_NSUB];
  __shared__ int red_i[4][TC_NSUB];
  for (int c0 = 0; c0 < N; c0 += 16) {
    float v[16], u2[16];
    tmem_ld16(trow + c0, v);
    if (DUAL) tmem_ld16(trow + TC_MAXN + c0, u2);
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
    if (!have) continue;
    if (P.epi == TC_ARGMAX) {
      // per column: max over the tile's 128 rows, lowest row on ties
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        float bv = v[j] * sc;
        int bi = P.row0 + wrow + m;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
          const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
          if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
        }
        if (lane == 0) { red_v[warp][(c0 + j) % TC_NSUB] = bv; red_i[warp][(c0 + j) % TC_NSUB] = bi; }
      }
      if ((c0 + 16) % TC_NSUB == 0 || c0 + 16 >= N) {
        __syncwarp();
        asm volatile("bar.sync 1, 128;" ::: "memory");
        const int cb = c0 + 16 - TC_NSUB < 0 ? 0 : (c0 + 16 - TC_NSUB);
        if (threadIdx.x < TC_NSUB) {
          const int c = cb + threadIdx.x;
          const int n = n0 + c;
          if (c < c0 + 16 && n < n0 + nrows) {
            float bv = red_v[0][threadIdx.x];
            int bi = red_i[0][threadIdx.x];
            for (int w = 1; w < 4; ++w) {
              const float ov = red_v[w][threadIdx.x];
              const int oi = red_i[w][threadIdx.x];
              if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
            }
            P.am_val[(size_t)(off + n) * P.am_ld + mt] = bv;
            P.am_idx[(size_t)(off + n) * P.am_ld + mt] = bi;
          }
        }
        asm volatile("bar.sync 1, 128;" ::: "memory");
      }
      continue;
    }
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int n = n0 + c0 + j;
      if (n >= n0 + nrows) break;
      const float val = v[j] * sc;
      const size_t r = (size_t)(off + n);
      if (P.epi == TC_STORE) {
        P.out_f32[r * P.ldo + col] = val;
      } else if (P.epi == TC_ADD) {
        P.out_f32[r * P.ldo + col] += val;
      } else if (P.epi == TC_SCATTER) {
        P.out_f32[(size_t)P.perm[r] * P.ldo + col] = val;
      } else if (DUAL && P.epi == TC_SWIGLU) {
        const float hv = silu(val) * (u2[j] * sc2);
        const uint16_t hi = f_to_bf16(hv);
        P.out_bf16[r * P.ldo + col] = hi;
        if (P.out_bf16_lo) P.out_bf16_lo[r * P.ldo + col] = f_to_bf16(hv - bf16_to_f(hi));
      }
    }
  }
  }   // warp < 4
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  if (warp == 1) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(NCOL));
}

// ---------------------------------------------------------------------------
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// 2D bf16 tensor map over rows of `inner` elements (row-major), box of
// 64 x box_rows, 128-byte swizzle, zero fill outside.
int tc_make_map(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return -1;
  if ((reinterpret_cast<uintptr_t>(base) & 15) || (inner * 2) % 16 || inner % TC_BK) return -2;
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {inner * 2};
  const cuuint32_t box[2] = {(cuuint32_t)TC_BK, box_rows};
  const cuuint32_t es[2] = {1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : -3;
}

// 2D e4m3 (byte) tensor map over rows of `inner` bytes, box of 64 x box_rows,
// no swizzle (the converters place the bytes).
int tc_make_map_u8(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return -1;
  if ((reinterpret_cast<uintptr_t>(base) & 15) || inner % 16 || inner % TC_BK) return -2;
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {inner};
  const cuuint32_t box[2] = {(cuuint32_t)TC_BK, box_rows};
  const cuuint32_t es[2] = {1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : -3;
}

}  // namespace spec

// ---------------------------------------------------------------------------
// Kernel-level entry point (tests and tools): with X = B (+ B_lo when given),
// out[n][m] = sum_k A[m][k] X[n][k] (dual = 0) or
// out_bf16[n][m] = silu(A[m]·X[n]) * (A2[m]·X[n]) (dual = 1).
// Kernel-level entry point (tests and tools): with X = B (+ B_lo when given)
// and weights A (bf16, or e4m3 when a_fp8, times the per-row scales),
// out[n][m] = sum_k A[m][k] X[n][k] (dual = 0) or
// out_bf16[n][m] = silu(A[m]·X[n]) * (A2[m]·X[n]) (dual = 1).
extern "C" int spec_tc_gemm_test(const void* a_dev, const void* a2_dev, const float* a_scale_dev,
                                 const float* a2_scale_dev, int a_fp8, const void* b_dev, const void* b_lo_dev,
                                 int M, int N, int K, int dual, void* out_dev, int* err_dev, uintptr_t cuda_stream) {
  using namespace spec;
  if (!a_dev || !b_dev || !out_dev || !err_dev || (dual && !a2_dev)) return set_last_error(-1, "null pointer");
  if (M < TC_BM || M % TC_BM || K < TC_BK || K % TC_BK || N < 1) return set_last_error(-1, "M, K multiples of 128, 64");
  static bool configured = false;
  if (!configured) {
    if (configure_tc_kernels() != cudaSuccess) return set_last_error(-3, "tc kernel attributes");
    configured = true;
  }
  TcMaps maps;
  maps.dual = dual;
  maps.f8 = a_fp8 ? 1 : 0;
  auto amap = [&](CUtensorMap* mp, const void* p) {
    return a_fp8 ? tc_make_map_u8(mp, p, K, M, TC_BM) : tc_make_map(mp, p, K, M, TC_BM);
  };
  if (amap(&maps.a, a_dev) || (dual && amap(&maps.a2, a2_dev)) || tc_make_map(&maps.b, b_dev, K, N, TC_NSUB) ||
      (b_lo_dev && tc_make_map(&maps.blo, b_lo_dev, K, N, TC_NSUB)))
    return set_last_error(-6, "tensor map encoding failed");
  if (!dual) maps.a2 = maps.a;
  if (!b_lo_dev) maps.blo = maps.b;
  TcParams P = {};
  P.K = K; P.Mg = M; P.N = N; P.ldo = M; P.epi = dual ? TC_SWIGLU : TC_STORE;
  P.out_f32 = dual ? nullptr : reinterpret_cast<float*>(out_dev);
  P.out_bf16 = dual ? reinterpret_cast<uint16_t*>(out_dev) : nullptr;
  P.scale = a_scale_dev;
  P.scale2 = a2_scale_dev;
  P.err = err_dev;
  P.split = b_lo_dev != nullptr;
  launch_tc_gemm(maps, P, M / TC_BM, 1, (N + TC_MAXN - 1) / TC_MAXN, reinterpret_cast<cudaStream_t>(cuda_stream));
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? 0 : set_last_error(-3, cudaGetErrorString(e));
}

namespace spec {

cudaError_t configure_tc_kernels() {
  cudaError_t e = cudaSuccess, r;
#define ALLOW(D, F)                                                                                        \
  if ((r = cudaFuncSetAttribute(k_tc_gemm<D, F>, cudaFuncAttributeMaxDynamicSharedMemorySize,             \
                                tc_smem_bytes(D, F))) != cudaSuccess)                                      \
    e = r
  ALLOW(0, 0); ALLOW(1, 0); ALLOW(0, 1); ALLOW(1, 1);
#undef ALLOW
  return e;
}

void launch_tc_gemm(const TcMaps& maps, const TcParams& P, int m_tiles, int groups, int n_tiles, cudaStream_t st) {
  const dim3 grid(m_tiles, groups, n_tiles);
  const CUtensorMap& a2 = maps.dual ? maps.a2 : maps.a;
  if (maps.f8) {
    if (maps.dual) k_tc_gemm<1, 1><<<grid, tc_threads(1), tc_smem_bytes(1, 1), st>>>(maps.a, a2, maps.b, maps.blo, P);
    else k_tc_gemm<0, 1><<<grid, tc_threads(1), tc_smem_bytes(0, 1), st>>>(maps.a, a2, maps.b, maps.blo, P);
  } else {
    if (maps.dual) k_tc_gemm<1, 0><<<grid, tc_threads(0), tc_smem_bytes(1, 0), st>>>(maps.a, a2, maps.b, maps.blo, P);
    else k_tc_gemm<0, 0><<<grid, tc_threads(0), tc_smem_bytes(0, 0), st>>>(maps.a, a2, maps.b, maps.blo, P);
  }
}

}  // namespace spec
