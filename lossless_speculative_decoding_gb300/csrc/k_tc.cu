// Tensor-core (tcgen05) GEMM for verify steps and prefill at T >= 16 rows.
//
// D[m, n] = sum_k W[m, k] * X[n, k]: weights W (bf16, row-major = K-major)
// fill the MMA's M = 128 rows, activation rows X its N <= 128 columns, so a
// CTA streams one 128-row weight tile once for all of its tokens. The
// activations are given as two bf16 operands, X = X_hi + X_lo (about 16
// mantissa bits): one MMA takes the hi rows and then the lo rows as its N
// columns and the epilogue adds the two, so the result keeps near-fp32
// activation precision while the weights stay exact bf16. Weights are stored
// pre-tiled (tc_pack_weights): every 128-row x 64-element tile (an atom) is
// one contiguous 16 KB block holding the exact 128-byte-swizzled shared-memory
// image, and the atoms of a row tile follow each other along K, so a stage
// fetches its one or two atoms with a single linear bulk copy
// (cp.async.bulk) instead of 128 strided row pieces; activation tiles
// come by TMA (cp.async.bulk.tensor, 128-byte swizzle). Stages run through a
// multi-stage mbarrier pipeline as deep as shared memory allows; one thread issues tcgen05.mma into a TMEM
// accumulator (fp32, lane = weight row, column = token); four warps read it
// back with tcgen05.ld for the epilogue. Experts are groups: the activation
// rows of group g are rows [off_g, off_g + cnt_g) of a permuted buffer, and a
// CTA computes the columns of one group, so each token column only ever sees
// its own row of X -- its result does not depend on the other tokens.
//
// FP8 weights (e4m3, per-row fp32 scale applied in the epilogue): the 8 KB
// e4m3 tile (row-major inside the tile) lands in the stage, eight converter
// warps widen it to f16 -- exactly, one conversion per pair of values -- into
// one of two 128-byte-swizzled operand buffers and signal the MMA thread, so
// the tensor cores run an f16 MMA while HBM carries one byte per weight. The
// activations of these GEMMs come as f16 parts of 256 x (hi + lo carry ~22
// significant bits); the epilogue divides the 256 back out. The widened tiles live in their own two-deep ring, not in the
// stages, so the stages (e4m3 + activations only) are small and many loads
// stay in flight.
//
// Every wait on an mbarrier ends by a deadline read from %globaltimer (or as
// soon as another CTA has reported a timeout); a timeout sets an error bit,
// the CTA stops issuing work, waits (to the deadline) for the copies and MMAs
// it has in flight, frees its TMEM and returns.
#include <cuda_fp8.h>
#include <algorithm>
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"
#include "spec.h"

namespace spec {

constexpr int TC_BM = 128;            // weight rows per CTA (MMA M)
constexpr int TC_BK = 64;             // K elements per atom (128 bytes of bf16, one swizzle row)
constexpr int TC_NSUB = 32;           // activation rows per TMA box
constexpr int TC_MAXN = 128;          // activation rows per CTA (largest N tile)
constexpr int TC_ACCW = 2 * TC_MAXN;  // TMEM columns of one accumulator (hi rows, then lo rows)
constexpr int TC_A_BYTES = TC_BM * TC_BK * 2;        // 16 KB
constexpr int TC_A8_BYTES = TC_BM * TC_BK;           // 8 KB e4m3 staging per weight operand

constexpr int TC_MAXST = 12;          // pipeline stages at most
constexpr int TC_SMEM = 220 * 1024;   // dynamic shared memory of every CTA
constexpr int TC_HDR = 1024;          // barriers + TMEM slot, ahead of the stages

constexpr int TC_NCONV_MAX = 4;       // FP8: widened weight buffers (converter -> MMA ring) at most

// Bytes of one pipeline stage of `at` K atoms for nsub 32-row activation
// boxes: the weight tile(s) as stored (bf16, or e4m3 staging for FP8) and the
// activation parts. Every part is a multiple of 1024 bytes, so each stays
// aligned for the 128-byte swizzle.
__host__ __device__ constexpr int tc_stage_bytes(int dual, int f8, int nsub, int split, int at) {
  return at * ((f8 ? TC_A8_BYTES : TC_A_BYTES) * (1 + dual) + (1 + split) * nsub * TC_NSUB * TC_BK * 2);
}
// FP8: widened buffers in the converter -> MMA ring. Two: a deeper ring
// costs TMA stages, and on the batch-64 e4m3 step three or four buffers for
// small activation tiles were slower (4.43 / 4.49 ms against 4.31 ms).
__host__ __device__ constexpr int tc_nconv(int f8, int /* nsub */) { return f8 ? 2 : 0; }
// FP8: the ring of widened bf16 weight tiles the MMAs read, after the stages.
__host__ __device__ constexpr int tc_conv_bytes(int dual, int f8, int nsub, int at) {
  return tc_nconv(f8, nsub) * at * TC_A_BYTES * (1 + dual);
}
// Stages that fit: as many weight tiles in flight as shared memory allows.
__host__ __device__ constexpr int tc_stage_count(int dual, int f8, int nsub, int split, int at) {
  return (TC_SMEM - TC_HDR - 1024 - tc_conv_bytes(dual, f8, nsub, at)) / tc_stage_bytes(dual, f8, nsub, split, at) <
                 TC_MAXST
             ? (TC_SMEM - TC_HDR - 1024 - tc_conv_bytes(dual, f8, nsub, at)) / tc_stage_bytes(dual, f8, nsub, split, at)
             : TC_MAXST;
}
// K atoms per stage: two (half the barrier round trips per weight byte)
// where three such stages still fit, else one.
__host__ __device__ constexpr int tc_atoms(int dual, int f8, int nsub, int split) {
  return tc_stage_count(dual, f8, nsub, split, 2) >= 3 ? 2 : 1;
}
__host__ __device__ constexpr int tc_threads(int f8) { return f8 ? 320 : 128; }

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

// Shared-memory matrix descriptor of a K-major bf16 tile stored as 128-byte
// rows with the 128-byte swizzle (8-row groups 1024 bytes apart). The start
// address sits in the low 14 bits (16-byte units) and shared addresses stay
// below 256 KB, so the descriptor of address + o is this one + o / 16.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);   // start address
  d |= (uint64_t)1 << 16;                      // leading byte offset (unused with this swizzle)
  d |= (uint64_t)(1024 >> 4) << 32;            // stride byte offset: 8 rows x 128 bytes
  d |= (uint64_t)1 << 46;                      // descriptor version
  d |= (uint64_t)2 << 61;                      // 128-byte swizzle
  return d;
}

// Instruction descriptor: bf16 x bf16 (f16 x f16 with f16) -> fp32, both operands K-major.
__device__ __forceinline__ uint32_t tc_idesc(int N, int f16) {
  const uint32_t ab = f16 ? 0u : 1u;                  // operand format: 0 f16, 1 bf16
  return (1u << 4) | (ab << 7) | (ab << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(TC_BM >> 4) << 24);
}

__device__ __forceinline__ void tma_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar) : "memory");
}

// 2^x by the hardware approximation (ex2.approx: relative error ~2^-22).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Linear global -> shared copy completing on an mbarrier (16-byte aligned, size a multiple of 16).
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
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

// Eight e4m3 values (one 8-byte word pair) as eight f16 values, exactly (one
// conversion per pair; every e4m3 value is an f16 normal or zero).
__device__ __forceinline__ uint4 e4m3x8_to_f16x8(uint2 v) {
  const uint32_t w[2] = {v.x, v.y};
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)((w[i] >> (16 * h)) & 0xFFFF), __NV_E4M3);
      o[2 * i + h] = (uint32_t)hr.x | ((uint32_t)hr.y << 16);
    }
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
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

constexpr int TC_NCONVW = 8;          // FP8 converter warps (warps 2..9: two on each SM sub-partition)

// Stage s of the FP8 form: e4m3 staging [128 rows][64 B] -> f16 tile [128
// rows][128 B] with the 128-byte swizzle (16-byte piece c of row r at
// (c ^ (r % 8)) * 16). The converter threads take the 1024 pieces round
// robin; a thread loads all its pieces before widening any.
__device__ __forceinline__ void convert_tile(const unsigned char* stg, unsigned char* dst, int t) {
  constexpr int NT = TC_NCONVW * 32, NI = (1024 + NT - 1) / NT;
  uint2 v[NI];
#pragma unroll
  for (int j = 0; j < NI; ++j) {
    const int i = t + NT * j, r = i >> 3, c = i & 7;
    if (i < 1024) v[j] = *reinterpret_cast<const uint2*>(stg + r * 64 + c * 8);
  }
#pragma unroll
  for (int j = 0; j < NI; ++j) {
    const int i = t + NT * j, r = i >> 3, c = i & 7;
    if (i < 1024) *reinterpret_cast<uint4*>(dst + r * 128 + ((c ^ (r & 7)) << 4)) = e4m3x8_to_f16x8(v[j]);
  }
}

template <int DUAL, int F8>
__global__ void __launch_bounds__(tc_threads(F8), 1) k_tc_gemm(const __grid_constant__ CUtensorMap mapB,
                                                               const __grid_constant__ CUtensorMap mapBlo,
                                                               const __grid_constant__ CUtensorMap mapBlo2, TcParams P) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  // header: full[MAXST], empty[MAXST], done, cfull[MAXST] (F8: widened tile ready; the first
  // NCV used), cempty[TC_NCONV_MAX] (F8: widened buffer free), TMEM slot, abort flag
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
  uint64_t* cempty = bars + 3 * TC_MAXST + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(cempty + TC_NCONV_MAX);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- the CTA's group and columns (whole-CTA early exits happen before any set-up) ----
  // N tiles vary fastest (CTAs sharing a weight tile run together); z = group x K split
  const int ksn = P.ksplit > 1 ? P.ksplit : 1;
  const int nt = blockIdx.x, mt = blockIdx.y, slot = blockIdx.z / ksn, ks = blockIdx.z % ksn;
  const int n_groups = P.g_n ? *P.g_n : (int)gridDim.z / ksn;
  if (slot >= n_groups) return;
  const int grp = P.g_expert ? P.g_expert[slot] : slot;
  const int off = P.g_off ? P.g_off[slot] : 0;
  const int cnt = P.g_cnt ? P.g_cnt[slot] : P.N;
  const int ntile = P.ntile;
  const int n0 = nt * ntile;
  if (n0 >= cnt) return;
  const int nrows = min(ntile, cnt - n0);
  const int nsub = (nrows + TC_NSUB - 1) / TC_NSUB;
  const int N = nsub * TC_NSUB;                       // activation rows: multiple of 32, <= 128
  const int NP = (1 + P.split) * N;                   // MMA N: the hi rows, then the lo (and lo2) rows
  // stage layout, AT K atoms per stage: bf16: [A atoms][A2 atoms (DUAL)][B
  // atoms, each hi rows then lo (lo2) rows]; FP8: [B atoms][e4m3 A atoms, A2
  // atoms], the widened tiles in the ring after the stages. The lo box follows
  // the hi box at N x 128 bytes (a whole number of 8-row swizzle groups), so
  // one MMA with N = NP multiplies the weights into all parts.
  const int AT = tc_atoms(DUAL, F8, nsub, P.split);
  const int BB = N * TC_BK * 2;                       // one activation part of one atom
  const int BAT = (1 + P.split) * BB;                 // one B atom
  const int SB = tc_stage_bytes(DUAL, F8, nsub, P.split, AT);
  const int STAGES = tc_stage_count(DUAL, F8, nsub, P.split, AT);
  const int BOFF = F8 ? 0 : AT * TC_A_BYTES * (1 + DUAL);
  const int STG_OFF = BOFF + AT * BAT;
  const int CONV_ONE = AT * TC_A_BYTES * (1 + DUAL);  // one widened buffer (FP8)
  unsigned char* stages = smem + TC_HDR;
  const int NCV = tc_nconv(F8, nsub);                 // FP8: widened buffers in the ring
  unsigned char* conv = stages + STAGES * SB;         // FP8: NCV widened buffers
  // this split's K atoms [kt0, kt1) (the host picks splits that are never empty)
  const int KTall = P.K / TC_BK, KTs = (KTall + ksn - 1) / ksn;
  const int kt0 = ks * KTs, kt1 = min(KTall, kt0 + KTs), KT = kt1 - kt0;
  const int NST = (KT + AT - 1) / AT;                 // stages of this CTA
  const int wrow = grp * P.Mg + mt * TC_BM;           // first weight row of the tile
  // Independent accumulators, so consecutive MMAs do not wait on each other:
  // accumulator kb takes the 16-wide K steps k with k % NKB == kb, columns
  // [0, N) the hi and [N, 2N) the lo activations; the epilogue adds (hi, kb 0),
  // (hi, kb 1), (lo, kb 0), (lo, kb 1) in that order. Accumulator kb of
  // matrix mat starts at column (mat * NKB + kb) * TC_ACCW.
  constexpr int NKB = DUAL ? 1 : 2;
  constexpr int NACC = 3 * NKB;                       // accumulators read back at most (three parts)
  constexpr uint32_t NCOL = 512;                      // TMEM columns: (1 + DUAL) * NKB * TC_ACCW

  // barrier indices: full s, empty TC_MAXST + s, done 2 TC_MAXST, cfull 2 TC_MAXST + 1 + c
  if (threadIdx.x == 0) {
    for (int i = 0; i < 2 * TC_MAXST + 1; ++i)
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(bars + i)));
    for (int i = 0; i < TC_MAXST; ++i)    // one arrival per converter warp
      asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bars + 2 * TC_MAXST + 1 + i)),
                   "r"(TC_NCONVW));
    for (int i = 0; i < TC_NCONV_MAX; ++i)    // one MMA commit
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(cempty + i)));
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
    constexpr int AST = F8 ? TC_A8_BYTES : TC_A_BYTES;
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&mapB)) : "memory");
    if (P.split > 0) asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&mapBlo)) : "memory");
    if (P.split > 1) asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&mapBlo2)) : "memory");
    // P.test_stall: issue nothing, so every wait on these copies runs to its
    // deadline (the check of the bounded waits)
    for (int i = 0; i < (P.test_stall ? 0 : NST); ++i) {
      const int a0 = i * AT, na = min(AT, KT - a0), s = i % STAGES;
      if (i >= STAGES && !mbar_wait_deadline(smem_u32(bars + TC_MAXST + s), ((i / STAGES) - 1) & 1, P.err)) {
        atomicOr(P.err, DERR_TIMEOUT);
        *abort_flag = 1;
        // shared memory must outlive the copies already issued: wait (to the
        // deadline, whatever other CTAs report) for each stage still in flight
        for (int j = i - STAGES; j < i; ++j)
          if (j >= 0) mbar_wait_deadline(smem_u32(bars + j % STAGES), (j / STAGES) & 1, nullptr);
        break;
      }
      unsigned char* st = stages + s * SB;
      const uint32_t full = smem_u32(bars + s);
      const uint32_t bytes = (uint32_t)na * (AST * (1 + DUAL) + BAT);
      asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(full), "r"(bytes) : "memory");
      // the stage's atoms of a row tile are contiguous in the pre-tiled weights
      unsigned char* at = F8 ? st + STG_OFF : st;
      const size_t toff = ((size_t)(wrow / TC_BM) * KTall + kt0 + a0) * AST;
      bulk_g2s(smem_u32(at), static_cast<const unsigned char*>(P.wa) + toff, na * AST, full);
      if (DUAL) bulk_g2s(smem_u32(at + AT * AST), static_cast<const unsigned char*>(P.wa2) + toff, na * AST, full);
      for (int j = 0; j < na; ++j) {
        unsigned char* bt = st + BOFF + j * BAT;
        const int kx = (kt0 + a0 + j) * TC_BK;
        for (int q = 0; q < nsub; ++q) {
          tma_2d(smem_u32(bt + q * TC_NSUB * TC_BK * 2), &mapB, kx, off + n0 + q * TC_NSUB, full);
          if (P.split > 0) tma_2d(smem_u32(bt + BB + q * TC_NSUB * TC_BK * 2), &mapBlo, kx, off + n0 + q * TC_NSUB, full);
          if (P.split > 1)
            tma_2d(smem_u32(bt + 2 * BB + q * TC_NSUB * TC_BK * 2), &mapBlo2, kx, off + n0 + q * TC_NSUB, full);
        }
      }
    }
  } else if (warp == 1 && lane == 0) {
    // ---- MMA issuer ----
    const uint32_t idesc = tc_idesc(NP, F8);
    const uint64_t d0 = sw128_desc(smem_u32(stages));
    bool ok = true;
    int kstep = 0;                                    // 16-wide K steps issued so far
    for (int i = 0; i < NST && ok; ++i) {
      const int s = i % STAGES, na = min(AT, KT - i * AT), c = F8 ? i % NCV : 0;
      // bf16: the TMA bytes of the stage; F8: the converters' signal for widened buffer c
      const bool arrived = F8 ? mbar_wait_deadline(smem_u32(bars + 2 * TC_MAXST + 1 + c), (i / NCV) & 1, P.err)
                              : mbar_wait_deadline(smem_u32(bars + s), (i / STAGES) & 1, P.err);
      if (!arrived) {
        atomicOr(P.err, DERR_TIMEOUT);
        *abort_flag = 1;
        ok = false;
        break;
      }
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const uint64_t ds = d0 + (uint64_t)((s * SB) >> 4);
      const uint64_t dsa = F8 ? sw128_desc(smem_u32(conv + c * CONV_ONE)) : ds;   // the weight tiles
      for (int j = 0; j < na; ++j) {
        const uint64_t da = dsa + (uint64_t)((j * TC_A_BYTES) >> 4);
        const uint64_t db = ds + (uint64_t)((BOFF + j * BAT) >> 4);
#pragma unroll
        for (int k = 0; k < TC_BK / 16; ++k, ++kstep) {
          const uint32_t acc = kstep >= NKB ? 1u : 0u;   // first MMA of an accumulator overwrites
          const uint32_t col = (uint32_t)((kstep % NKB) * TC_ACCW);
          asm volatile(
              "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
              " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n"
              ::"r"(tmem + col), "l"(da + 2 * k), "l"(db + 2 * k), "r"(idesc), "r"(acc));
          if (DUAL)
            asm volatile(
                "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
                " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n"
                ::"r"(tmem + (uint32_t)(NKB * TC_ACCW) + col), "l"(da + (uint64_t)((AT * TC_A_BYTES) >> 4) + 2 * k),
                  "l"(db + 2 * k), "r"(idesc), "r"(acc));
        }
      }
      asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                   ::"r"(smem_u32(bars + TC_MAXST + s)) : "memory");
      if (F8)   // widened buffer c is free once these MMAs complete
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                     ::"r"(smem_u32(cempty + c)) : "memory");
    }
    // "done" fires once every MMA issued so far has completed -- also after an
    // abort, so TMEM is never freed under an MMA in flight
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 ::"r"(smem_u32(bars + 2 * TC_MAXST)) : "memory");
  } else if (F8 && warp >= 2) {
    // ---- converters (warps 2..9): e4m3 staging -> swizzled f16 operand tile ----
    const int t = threadIdx.x - 64;
    for (int i = 0; i < NST; ++i) {
      const int s = i % STAGES, na = min(AT, KT - i * AT), c = i % NCV;
      if (!mbar_wait_deadline(smem_u32(bars + s), (i / STAGES) & 1, P.err) ||
          (i >= NCV && !mbar_wait_deadline(smem_u32(cempty + c), ((i / NCV) - 1) & 1, P.err))) {
        if (lane == 0) atomicOr(P.err, DERR_TIMEOUT);
        break;
      }
      unsigned char* st = stages + s * SB;
      unsigned char* cv = conv + c * CONV_ONE;
      for (int j = 0; j < na; ++j) {
        convert_tile(st + STG_OFF + j * TC_A8_BYTES, cv + j * TC_A_BYTES, t);
        if (DUAL) convert_tile(st + STG_OFF + (AT + j) * TC_A8_BYTES, cv + (AT + j) * TC_A_BYTES, t);
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0)
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bars + 2 * TC_MAXST + 1 + c)) : "memory");
    }
  }
  __syncwarp();

  // ---- epilogue: warp w holds TMEM lanes 32w..32w+31 = weight rows ----
  const bool done = mbar_wait_deadline(smem_u32(bars + 2 * TC_MAXST), 0, nullptr);
  const bool have = __syncthreads_and(done && *abort_flag == 0) != 0;   // block-uniform
  if (!have && threadIdx.x == 0) atomicOr(P.err, DERR_TIMEOUT);
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const int m = warp * 32 + lane;                     // row within the tile
  const int col = mt * TC_BM + m;                     // output feature (row within the group)
  // e4m3 weights multiply f16 parts of 256 x: the epilogue takes the 256 out (exactly)
  const float osc = F8 ? 1.0f / F16_OP_SCALE : 1.0f;
  const float sc = ((P.scale && have && warp < 4) ? P.scale[wrow + m] : 1.f) * osc;
  const float sc2 = ((DUAL && P.scale2 && have && warp < 4) ? P.scale2[wrow + m] : 1.f) * osc;
  const uint32_t trow = tmem + ((uint32_t)((warp & 3) * 32) << 16);
  __shared__ float red_v[4][TC_NSUB];
  __shared__ int red_i[4][TC_NSUB];
  __shared__ int s_last;
  // v = sum of the used accumulators in order (part 0 kb 0, part 0 kb 1, part 1 ...)
  auto load_acc = [&](int c0, float (&v)[16], float (&u2)[16]) {
    float t[NACC][16], t2[NACC][16];
    const int nacc = (1 + P.split) * NKB;
#pragma unroll
    for (int a = 0; a < NACC; ++a) {
      if (a < nacc) {
        const uint32_t c = (uint32_t)((a % NKB) * TC_ACCW + (a / NKB) * N + c0);   // (part a / NKB, kb a % NKB)
        tmem_ld16(trow + c, t[a]);
        if (DUAL) tmem_ld16(trow + (uint32_t)(NKB * TC_ACCW) + c, t2[a]);
      }
    }
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      float x = t[0][j], y = DUAL ? t2[0][j] : 0.f;
#pragma unroll
      for (int a = 1; a < NACC; ++a) {
        if (a < nacc) {
          x += t[a][j];
          if (DUAL) y += t2[a][j];
        }
      }
      v[j] = x;
      u2[j] = y;
    }
  };
  // the epilogue of columns c0..c0+15 (warps 0-3)
  auto emit = [&](int c0, const float (&v)[16], const float (&u2)[16]) {
    if (P.epi == TC_ARGMAX) {
      // per column: max over the tile's 128 rows, lowest row on ties
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        float bv = am_key(v[j] * sc);
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
      return;
    }
    if (P.epi == TC_ADD) {
      // all sixteen residual values are loaded before any store (a load-add-
      // store chain would wait for each round trip in turn)
      float old[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int n = n0 + c0 + j;
        old[j] = n < n0 + nrows ? P.out_f32[(size_t)(off + n) * P.ldo + col] : 0.f;
      }
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int n = n0 + c0 + j;
        if (n < n0 + nrows) P.out_f32[(size_t)(off + n) * P.ldo + col] = old[j] + v[j] * sc;
      }
      return;
    }
    if (P.epi == TC_SCATTER) {
      int dst[16];   // destination rows, all loaded before the first store
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int n = n0 + c0 + j;
        dst[j] = n < n0 + nrows ? P.perm[off + n] : -1;
      }
#pragma unroll
      for (int j = 0; j < 16; ++j)
        if (dst[j] >= 0) P.out_f32[(size_t)dst[j] * P.ldo + col] = v[j] * sc;
      return;
    }
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int n = n0 + c0 + j;
      if (n >= n0 + nrows) break;
      const float val = v[j] * sc;
      const size_t r = (size_t)(off + n);
      if (P.epi == TC_STORE) {
        P.out_f32[r * P.ldo + col] = val;
      } else if (DUAL && P.epi == TC_SWIGLU) {
        const float hv = silu(val) * (u2[j] * sc2);
        uint16_t pp[2];
        split_parts(hv, F8, 2, pp);                    // operand parts of the (same-format) down GEMM
        P.out_bf16[r * P.ldo + col] = pp[0];
        if (P.out_bf16_lo) P.out_bf16_lo[r * P.ldo + col] = pp[1];
      }
    }
  };
  if (ksn == 1 && (P.epi == TC_ARGMAX || P.epi == TC_STATS) && TC_BM * (N + 1) * 4 <= STAGES * SB) {
    // per column: max over the tile's 128 rows, lowest row on ties. Every MMA
    // has completed and every copy has landed, so the stage memory holds the
    // [row][column] values (row stride N + 1: conflict-free both ways) and one
    // thread per column scans its rows -- no chain of warp shuffles
    float* tv = reinterpret_cast<float*>(stages);
    const int LD = N + 1;
    if (warp < 4) {
      for (int c0 = 0; c0 < N; c0 += 16) {
        float v[16], u2[16];
        load_acc(c0, v, u2);
#pragma unroll
        for (int j = 0; j < 16; ++j) tv[m * LD + c0 + j] = P.epi == TC_ARGMAX ? am_key(v[j] * sc) : v[j] * sc;
      }
    }
    __syncthreads();
    const int n = threadIdx.x;
    if (P.epi == TC_STATS && have && n < nrows) {
      // column n: the tile's max of x * it, then sum of exp(x * it - max) as
      // 2^(x it log2 e - max log2 e) in row order; again without the row's
      // draft when it lies in the tile (its logit goes to xd)
      const StatsOut& so = P.st;
      const int t = off + n0 + n;
      const float it = *so.it;
      float mx = -INFINITY;
      for (int r = 0; r < TC_BM; ++r) mx = fmaxf(mx, tv[r * LD + n]);
      const float mm = mx * it, cl = it * 1.4426950408889634f, mb = mm * 1.4426950408889634f;
      float sum = 0.f;
      for (int r = 0; r < TC_BM; ++r) sum += ex2_approx(fmaf(tv[r * LD + n], cl, -mb));
      const int sq = t / so.R, j = t % so.R;
      const int nd = min(max(so.nd[sq], 0), so.K);
      const int local = j < nd ? so.drafts[sq * so.K + j] - (P.row0 + wrow) : -1;
      float sk = sum;
      if (local >= 0 && local < TC_BM) {
        sk = 0.f;
        for (int r = 0; r < TC_BM; ++r)
          if (r != local) sk += ex2_approx(fmaf(tv[r * LD + n], cl, -mb));
        so.xd[t] = tv[local * LD + n];
      }
      float* o = so.out + ((size_t)t * P.am_ld + mt) * 4;
      *reinterpret_cast<float4*>(o) = make_float4(mm, sum, sk, 0.f);
    } else if (have && n < nrows) {
      float bv[4];
      int bi[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) { bv[u] = tv[u * LD + n]; bi[u] = u; }
      for (int r = 4; r < TC_BM; r += 4) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float c = tv[(r + u) * LD + n];
          if (c > bv[u]) { bv[u] = c; bi[u] = r + u; }        // rows in increasing order: ties keep the lower
        }
      }
#pragma unroll
      for (int u = 1; u < 4; ++u)
        if (bv[u] > bv[0] || (bv[u] == bv[0] && bi[u] < bi[0])) { bv[0] = bv[u]; bi[0] = bi[u]; }
      P.am_val[(size_t)(off + n0 + n) * P.am_ld + mt] = bv[0];
      P.am_idx[(size_t)(off + n0 + n) * P.am_ld + mt] = P.row0 + wrow + bi[0];
    }
  } else if (ksn == 1) {
    if (warp < 4) {
      for (int c0 = 0; c0 < N; c0 += 16) {
        float v[16], u2[16];
        load_acc(c0, v, u2);
        if (have) emit(c0, v, u2);
      }
    }
  } else {
    // split K: every split stores its fp32 partial [split][part][row][feature];
    // the last split of the tile to arrive adds them in split order and runs
    // the epilogue (the order does not depend on which split came last)
    const size_t pstride = (size_t)P.part_n * P.part_m;
    const size_t feat = (size_t)wrow + m;
    if (warp < 4) {
      for (int c0 = 0; c0 < N; c0 += 16) {
        float v[16], u2[16];
        load_acc(c0, v, u2);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int n = n0 + c0 + j;
          if (n >= n0 + nrows) break;
          const size_t e = (size_t)(off + n) * P.part_m + feat;
          P.part[(size_t)ks * (1 + DUAL) * pstride + e] = v[j];
          if (DUAL) P.part[((size_t)ks * 2 + 1) * pstride + e] = u2[j];
        }
      }
    }
    __threadfence();
    __syncthreads();
    const int tile = ((slot * (int)gridDim.y) + mt) * (int)gridDim.x + nt;
    if (threadIdx.x == 0) s_last = atomicAdd(P.tile_cnt + tile, 1) == ksn - 1;
    __syncthreads();
    if (s_last) {
      __threadfence();
      if (warp < 4 && have) {
        for (int c0 = 0; c0 < N; c0 += 16) {
          float v[16], u2[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) v[j] = u2[j] = 0.f;
          // split by split, the sixteen columns' loads are all issued before
          // any add (one round trip per split, not per column and split)
          for (int q = 0; q < ksn; ++q) {
            const float* pq = P.part + (size_t)q * (1 + DUAL) * pstride + feat;
            float t[16], t2[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int n = n0 + c0 + j;
              const size_t e = (size_t)(off + n) * P.part_m;
              t[j] = n < n0 + nrows ? __ldcg(pq + e) : 0.f;
              t2[j] = DUAL && n < n0 + nrows ? __ldcg(pq + pstride + e) : 0.f;
            }
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              v[j] += t[j];
              if (DUAL) u2[j] += t2[j];
            }
          }
          emit(c0, v, u2);
        }
      }
      if (threadIdx.x == 0) P.tile_cnt[tile] = 0;
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  if (warp == 1) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(NCOL));
}

// ---------------------------------------------------------------------------
// Weight tiling: W [rows, K] row-major -> tiles (row tile R, K tile kt) in
// order R * (K / 64) + kt. bf16: 16 KB per tile, row r's 16-byte piece c at
// r * 128 + (c ^ (r % 8)) * 16 (the 128-byte swizzle); e4m3: 8 KB per tile,
// row r's piece c at r * 64 + c * 16. One thread per 16-byte piece.
__global__ void k_pack_weights(const uint4* __restrict__ src, uint4* __restrict__ dst, int rows, int K, int f8) {
  const int ppr = f8 ? K / 16 : K / 8;                 // 16-byte pieces per row
  const int ppt = f8 ? 4 : 8;                          // pieces per row inside a tile
  const int KT = K / TC_BK;
  const size_t n = (size_t)rows * ppr;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    const int row = (int)(i / ppr), pc = (int)(i % ppr);
    const int R = row / TC_BM, r = row % TC_BM, kt = pc / ppt, c = pc % ppt;
    const size_t tile = (size_t)R * KT + kt;
    const size_t piece = f8 ? tile * (TC_A8_BYTES / 16) + (size_t)r * 4 + c
                            : tile * (TC_A_BYTES / 16) + (size_t)r * 8 + (c ^ (r & 7));
    dst[piece] = src[i];
  }
}

bool tc_column_scan_fits(int rows) {
  const int nsub = (rows + TC_NSUB - 1) / TC_NSUB, N = nsub * TC_NSUB;
  const int at = tc_atoms(0, 0, nsub, 1);
  return TC_BM * (N + 1) * 4 <= tc_stage_count(0, 0, nsub, 1, at) * tc_stage_bytes(0, 0, nsub, 1, at);
}

int tc_pack_weights(void* dst, const void* src, int rows, int K, int f8, cudaStream_t st) {
  if (rows % TC_BM || K % TC_BK || (reinterpret_cast<uintptr_t>(dst) & 15) || (reinterpret_cast<uintptr_t>(src) & 15))
    return -1;
  const size_t pieces = (size_t)rows * (f8 ? K / 16 : K / 8);
  const int blocks = (int)std::min<size_t>((pieces + 255) / 256, 65535);
  k_pack_weights<<<blocks, 256, 0, st>>>(static_cast<const uint4*>(src), static_cast<uint4*>(dst), rows, K, f8);
  return cudaGetLastError() == cudaSuccess ? 0 : -3;
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

// 3D byte map over a stack of weight rows ([rows][K] of esz-byte elements,
// row-major) for the streamed GEMVs: dims (128 bytes, rows, K * esz / 128
// chunks) -- the chunk before the row in memory, after it in the map, so a
// box lands as [chunk][row][128 bytes] -- box 128 x box_rows x box_chunks,
// 128-byte swizzle.
int gemv_make_map(CUtensorMap* map, const void* base, int esz, uint64_t K, uint64_t rows, uint32_t box_rows,
                  uint32_t box_chunks) {
  auto fn = encode_fn();
  if (!fn) return -1;
  if ((reinterpret_cast<uintptr_t>(base) & 15) || (K * esz) % 128) return -2;
  const cuuint64_t dims[3] = {128, rows, K * esz / 128};
  const cuuint64_t strides[2] = {K * esz, 128};
  const cuuint32_t box[3] = {128, box_rows, box_chunks};
  const cuuint32_t es[3] = {1, 1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : -3;
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

int kv_make_map(CUtensorMap* map, const void* kv, int head_dim, int page_size, int planes, int n_pages,
                size_t page_elems) {
  auto fn = encode_fn();
  if (!fn) return -1;
  if ((reinterpret_cast<uintptr_t>(kv) & 15) || head_dim % 64 || page_size % 16) return -2;
  const int halves = head_dim / 64;
  // key before half: a box lands in shared memory as [plane][half][key][64],
  // so the 128-byte rows of consecutive keys take consecutive swizzle phases
  const cuuint64_t dims[5] = {64, (cuuint64_t)page_size, (cuuint64_t)halves, (cuuint64_t)planes,
                              (cuuint64_t)n_pages};
  const cuuint64_t strides[4] = {(cuuint64_t)head_dim * 2, 128, (cuuint64_t)page_size * head_dim * 2,
                                 (cuuint64_t)page_elems * 2};
  const cuuint32_t box[5] = {64, (cuuint32_t)(page_size % 64 == 0 ? 64 : 16), (cuuint32_t)halves, 2, 1};
  const cuuint32_t es[5] = {1, 1, 1, 1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(kv), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : -3;
}

}  // namespace spec

// ---------------------------------------------------------------------------
// Kernel-level entry point (tests and tools): with X = B (+ B_lo when given)
// and weights A (bf16, or e4m3 when a_fp8, times the per-row scales),
// out[n][m] = sum_k A[m][k] X[n][k] (dual = 0) or
// out_bf16[n][m] = silu(A[m]·X[n]) * (A2[m]·X[n]) (dual = 1).
extern "C" int spec_tc_gemm_test(const void* a_dev, const void* a2_dev, const float* a_scale_dev,
                                 const float* a2_scale_dev, int a_fp8, const void* b_dev, const void* b_lo_dev,
                                 int M, int N, int K, int dual, int n_tile, int k_split, int flags,
                                 void* out_dev, int* err_dev, uintptr_t cuda_stream) {
  using namespace spec;
  if (!a_dev || !b_dev || !out_dev || !err_dev || (dual && !a2_dev)) return set_last_error(-1, "null pointer");
  if (M < TC_BM || M % TC_BM || K < TC_BK || K % TC_BK || N < 1) return set_last_error(-1, "M, K multiples of 128, 64");
  if (n_tile == 0) n_tile = TC_MAXN;
  if (n_tile != 32 && n_tile != 64 && n_tile != 128) return set_last_error(-1, "n_tile: 32, 64 or 128");
  if (k_split < 1) k_split = 1;
  if (k_split > K / TC_BK) return set_last_error(-1, "k_split larger than the K tiles");
  {
    const int kts = (K / TC_BK + k_split - 1) / k_split;   // splits the kernel sees are never empty
    k_split = (K / TC_BK + kts - 1) / kts;
  }
  static bool configured = false;
  if (!configured) {
    if (configure_tc_kernels() != cudaSuccess) return set_last_error(-3, "tc kernel attributes");
    configured = true;
  }
  TcMaps maps;
  maps.dual = dual;
  maps.f8 = a_fp8 ? 1 : 0;
  if (tc_make_map(&maps.b, b_dev, K, N, TC_NSUB) || (b_lo_dev && tc_make_map(&maps.blo, b_lo_dev, K, N, TC_NSUB)))
    return set_last_error(-6, "tensor map encoding failed");
  if (!b_lo_dev) maps.blo = maps.b;
  maps.blo2 = maps.blo;
  // the weights in the tiled layout, in stream-ordered scratch
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(cuda_stream);
  const size_t wbytes = (size_t)M * K * (a_fp8 ? 1 : 2);
  void* wt[2] = {nullptr, nullptr};
  for (int i = 0; i < 1 + (dual ? 1 : 0); ++i) {
    if (cudaMallocAsync(&wt[i], wbytes, st) != cudaSuccess) return set_last_error(-5, "scratch allocation");
    if (tc_pack_weights(wt[i], i ? a2_dev : a_dev, M, K, a_fp8, st)) return set_last_error(-3, "weight tiling");
  }
  TcParams P = {};
  P.wa = wt[0];
  P.wa2 = dual ? wt[1] : wt[0];
  P.K = K; P.Mg = M; P.N = N; P.ldo = M; P.epi = dual ? TC_SWIGLU : TC_STORE;
  P.out_f32 = dual ? nullptr : reinterpret_cast<float*>(out_dev);
  P.out_bf16 = dual ? reinterpret_cast<uint16_t*>(out_dev) : nullptr;
  P.scale = a_scale_dev;
  P.scale2 = a2_scale_dev;
  P.err = err_dev;
  P.split = b_lo_dev != nullptr;
  P.ntile = n_tile;
  P.ksplit = k_split;
  P.test_stall = (flags & SPEC_TC_TEST_STALL) ? 1 : 0;
  const int n_tiles = (N + n_tile - 1) / n_tile;
  float* part = nullptr;
  int* cnt = nullptr;
  if (k_split > 1) {
    if (cudaMallocAsync(reinterpret_cast<void**>(&part), (size_t)k_split * (1 + dual) * N * M * sizeof(float), st) !=
            cudaSuccess ||
        cudaMallocAsync(reinterpret_cast<void**>(&cnt), (size_t)(M / TC_BM) * n_tiles * sizeof(int), st) != cudaSuccess)
      return set_last_error(-5, "scratch allocation");
    cudaMemsetAsync(cnt, 0, (size_t)(M / TC_BM) * n_tiles * sizeof(int), st);
    P.part = part; P.part_n = N; P.part_m = M; P.tile_cnt = cnt;
  }
  launch_tc_gemm(maps, P, M / TC_BM, k_split, n_tiles, st);
  for (int i = 0; i < 2; ++i)
    if (wt[i]) cudaFreeAsync(wt[i], st);
  if (part) cudaFreeAsync(part, st);
  if (cnt) cudaFreeAsync(cnt, st);
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? 0 : set_last_error(-3, cudaGetErrorString(e));
}

namespace spec {

cudaError_t configure_tc_kernels() {
  cudaError_t e = cudaSuccess, r;
#define ALLOW(D, F)                                                                                        \
  if ((r = cudaFuncSetAttribute(k_tc_gemm<D, F>, cudaFuncAttributeMaxDynamicSharedMemorySize,             \
                                TC_SMEM)) != cudaSuccess)                                                  \
    e = r
  ALLOW(0, 0); ALLOW(1, 0); ALLOW(0, 1); ALLOW(1, 1);
#undef ALLOW
  return e;
}

void launch_tc_gemm(const TcMaps& maps, const TcParams& P, int m_tiles, int groups, int n_tiles, cudaStream_t st) {
  const dim3 grid(n_tiles, m_tiles, groups);
  TcParams Q = P;
  if (Q.ntile == 0) Q.ntile = TC_MAXN;
  if (maps.f8) {
    if (maps.dual) k_tc_gemm<1, 1><<<grid, tc_threads(1), TC_SMEM, st>>>(maps.b, maps.blo, maps.blo2, Q);
    else k_tc_gemm<0, 1><<<grid, tc_threads(1), TC_SMEM, st>>>(maps.b, maps.blo, maps.blo2, Q);
  } else {
    if (maps.dual) k_tc_gemm<1, 0><<<grid, tc_threads(0), TC_SMEM, st>>>(maps.b, maps.blo, maps.blo2, Q);
    else k_tc_gemm<0, 0><<<grid, tc_threads(0), TC_SMEM, st>>>(maps.b, maps.blo, maps.blo2, Q);
  }
}

}  // namespace spec
