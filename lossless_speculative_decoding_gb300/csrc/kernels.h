// Internal launch interface of the verify-step kernels (not part of the C ABI).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace spec {

constexpr int ATT_CHUNK = 64;     // keys per split-KV chunk (fixed at absolute positions)
constexpr int ATT_MAX_GROUPS = 1024;   // row groups (sequence slices of <= 32 rows) per attention launch
constexpr int GEMV_TP = 4;        // activation rows per GEMV pass
constexpr int GEMV_WARPS = 8;     // warps per GEMV block
constexpr int GEMV_G = 4;         // 16-byte weight chunks loaded per lane before use

struct LayerW {
  const float* attn_norm;
  const void* w_qkv; const float* s_qkv;
  const void* w_o; const float* s_o;
  const float* ffn_norm;
  const void* w_router;
  const void* w_gate; const float* s_gate;
  const void* w_up; const float* s_up;
  const void* w_down; const float* s_down;
  // streamed expert GEMVs (<= 8 rows, bf16 / e4m3): tensor maps of w_gate,
  // w_up, w_down (null: the register form) and the K per stage of each
  const CUtensorMap* ffn_map;
  int kst_gu, kst_dn;
};

// Shapes and device state shared by every kernel of a model.
struct Dims {
  int L, h, Hq, Hkv, d, E, k, S, inter, V;
  int wdtype;            // 0 f32, 1 bf16, 2 fp8, 3 nvfp4 (attention + experts)
  int act_f32;           // KV cache / embeddings / LM head in f32 (else bf16)
  int op_f16;            // operands of the e4m3-weight tensor-core GEMMs are f16 parts of 256 x (else bf16 parts of x)
  int P;                 // page size
  int max_pages;         // block-table row length
  int max_ctx;
  int NS;                // slots per row = k + S
  int n_sm;              // streaming multiprocessors (persistent grids)
  float eps, theta;
  size_t page_elems;     // elements per KV page (all layers)
};

struct DevState {
  void* kv;              // [n_pages][L][Hkv][2 (K, V)][P][d]
  const int* bt;         // [slots][max_pages]
  int* seq_len;          // [slots]
  int* last_tok;         // [slots]
  int* keep_pages;       // [slots]
  int* out_tok;          // [slots][max_ctx]
  int* n_out;            // [slots]
  const float* rope_cos; // [max_ctx][d/2]
  const float* rope_sin;
  int* err;              // device error bits
};

// Per-step scratch (sized for the largest T the model runs).
struct StepBuf {
  int* row_tok; int* row_pos; int* row_seq; int* row_src;
  int* row_rope;     // RoPE position of a row when it differs from its cache index (null: the same)
  float* x;          // [T, h] residual stream
  float* q;          // [T, Hq, d]
  float* att_o;      // [T, Hq, n_chunk_max, d] partial outputs
  float* att_ml;     // [T, Hq, n_chunk_max, 2] partial (max, sum)
  float* o;          // [T, Hq*d]
  float* u;          // [T, h] normed FFN input
  int* ids; float* wts;              // [T, k]
  int* perm;                         // [T*NS] pair ids grouped by expert
  int* act_expert; int* act_off; int* act_cnt; int* n_active;  // active-expert list
  int* counter;                      // [0] router arrivals over rows, [1] argmax-commit block arrivals
                                     // (each kept at zero between launches)
  float* rlogit;                     // [Tmax, E] router logits
  int* cnt_row;                      // [Tmax] router arrivals per row (expert-group blocks)
  int* cnt_att;                      // [Tmax * Hkv] attention arrivals per (row group, kv head)
  int* cnt_lm;                       // [ceil(Tmax/TP)] LM-head arrivals per row pass
  float* h_act;      // [T*NS, inter]
  float* y;          // [T*NS, h]
  float* am_val; int* am_idx;        // [T, n_vocab_blocks] argmax partials
  int* g;            // [T] greedy tokens
  // tensor-core path operands (null when the model streams with SIMT GEMVs)
  float* qkv;             // [T, (Hq+2Hkv) d] QKV GEMM output
  // each bf16 operand X is stored as hi = bf16(X) and lo = bf16(X - hi)
  uint16_t* xn_bf16;      // [T, h] RMS-normalised rows
  uint16_t* xn_lo;
  uint16_t* xn_lo2;       // third part bf16(X - hi - lo) (QKV input: outputs rounded for the KV cache)
  uint16_t* o_bf16;       // [T, Hq d] attention output
  uint16_t* o_lo;
  uint16_t* xperm;        // [T*NS, h] FFN input rows in expert-permuted order
  uint16_t* xperm_lo;
  uint16_t* hperm;        // [T*NS, inter] SwiGLU output in expert-permuted order
  uint16_t* hperm_lo;
  int* step_in;      // staging: [seq ids (max_batch) | drafts (max_batch*K) | n_draft (max_batch)]
  int* step_out;     // staging: [acc (max_batch) | bonus (max_batch) | device error bits]
  unsigned long long* out_ptrs;  // [2] caller device outputs (acc, bonus) of a _dev step; 0 = none.
                                 // Lives just before step_in so one host copy refreshes both.
  int n_chunk_max;
  int n_vblocks;
  int max_batch;      // staging block capacity (sequences per step)
};

void launch_rope_table(const Dims& D, float* cos_t, float* sin_t, cudaStream_t st);
void launch_assemble_verify(const Dims& D, const DevState& S, const StepBuf& B, const void* tok_embed,
                            int n_seq, int K, cudaStream_t st);
void launch_assemble_prefill(const Dims& D, const DevState& S, const StepBuf& B, const void* tok_embed,
                             const void* vis, int seq, int pos0, int T, cudaStream_t st);
void launch_qkv(const Dims& D, const DevState& S, const StepBuf& B, const LayerW& W, int layer, int T,
                const float* x, cudaStream_t st);
bool attn_separate_merge(const Dims& D, int R, int T);   // merge as its own launch
int attn_groups(const Dims& D, int T, int R);
void launch_attn_part(const Dims& D, const DevState& S, const StepBuf& B, int layer, int T, int R,
                      const CUtensorMap& kvmap, cudaStream_t st);
void launch_oproj(const Dims& D, const StepBuf& B, const LayerW& W, int T, float* xres, cudaStream_t st);
// full: always compute top-k and the permutation (the tensor-core path needs them)
void launch_router(const Dims& D, const StepBuf& B, const LayerW& W, int T, const float* xres, bool full,
                   cudaStream_t st);
void launch_gateup(const Dims& D, const StepBuf& B, const LayerW& W, int T, int* err, cudaStream_t st);
// At small T the router kernel writes only logits and gate/up routes in its prologue.
bool route_in_gateup(int T);
void launch_down(const Dims& D, const StepBuf& B, const LayerW& W, int T, int* err, cudaStream_t st);
// In-place expert combine of the residual x.
void launch_combine(const Dims& D, const StepBuf& B, float* x, int T, cudaStream_t st);
void launch_lmhead(const Dims& D, const StepBuf& B, const void* lm_head, const float* final_norm,
                   const float* x, int T, float* logits_dbg, bool fuse_argmax, cudaStream_t st);
// Streaming LM head + argmax for the verify step / prefill; with commit, its
// last block also accepts and commits the n_seq sequences (K drafts each).
void launch_lmhead_step(const Dims& D, const DevState& S, const StepBuf& B, const void* lm_head,
                        const float* final_norm, const float* x, int T, float* logits_dbg, bool commit,
                        int n_seq, int K, cudaStream_t st);
int lmhead_step_warps(const Dims& D);
int ffn_stage_k(int K, int esz);
void launch_argmax(const StepBuf& B, int T, cudaStream_t st);

// ---- tensor-core GEMM (k_tc.cu) ---------------------------------------------
enum TcEpi { TC_STORE = 0, TC_SWIGLU = 1, TC_ADD = 2, TC_ARGMAX = 3, TC_SCATTER = 4, TC_STATS = 5 };

// TC_STATS (the LM head of a sampled step): per (row, 128-row tile of the
// vocabulary) the softmax statistics of logit * it -- the max m, sum of
// exp(x it - m), and the same sum without the row's draft -- and, from the
// tile holding the row's draft, the draft's logit. Rows are step rows s R + j;
// row j < n_draft[s] of sequence s has draft drafts[s K + j].
struct StatsOut {
  float* out;             // [rows][tiles][4]: m, sum, sum without the draft, 0
  float* xd;              // [rows]
  const float* it;        // 1 / temperature (device)
  const int* drafts;      // [n_seq][K]
  const int* nd;          // [n_seq]
  int K, R;
};

struct TcParams {
  const void* wa;         // weights, tiled by tc_pack_weights
  const void* wa2;        // second weights (SWIGLU up), tiled
  int K;                  // reduction length (multiple of 64)
  int Mg;                 // weight rows per group (multiple of 128)
  int N;                  // activation rows when not grouped
  int ldo;                // output row stride (elements)
  int epi;                // TcEpi
  int row0;               // added to the weight row in argmax candidates
  // groups (nullptr: group = blockIdx.y, rows [0, N))
  const int* g_expert;
  const int* g_off;
  const int* g_cnt;
  const int* g_n;
  float* out_f32;         // STORE [off+n][col] / ADD (+=) / SCATTER [perm[off+n]][col]
  uint16_t* out_bf16;     // SWIGLU [off+n][col] (hi part)
  uint16_t* out_bf16_lo;  // SWIGLU low part (value - hi), nullable
  int split;              // extra activation parts: 0 (one bf16 operand), 1 (hi + lo), 2 (hi + lo + lo2)
  int ntile;              // activation rows per CTA: 32, 64 or 128 (0: 128)
  int ksplit;             // K splits (grid z = groups x ksplit); > 1: partials in `part`, summed by the last split
  float* part;            // [ksplit][1 + dual][part_n][part_m] fp32 partials
  int part_n, part_m;     // activation rows / weight rows of the launch
  int* tile_cnt;          // per (group, m tile, n tile) arrival counters, zero between launches
  const int* perm;
  const float* scale;     // per weight row (nullable)
  const float* scale2;    // per weight row of the second operand (SWIGLU up)
  float* am_val;          // ARGMAX candidates [off+n][am_ld]
  int* am_idx;
  int am_ld;
  int* err;
  int test_stall;         // test only: the producer issues no copies, so every wait times out
  StatsOut st;            // TC_STATS outputs
};

struct TcMaps {
  CUtensorMap b, blo, blo2;    // activation parts hi, lo, lo2
  int dual;
  int f8 = 0;                  // weights are e4m3
};

// 2D bf16 tensor map: rows of `inner` elements, box 64 x box_rows, 128-byte
// swizzle. Returns 0 on success.
int tc_make_map(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint32_t box_rows);
// 5D bf16 tensor map over the paged KV pool [pages][layer][kv head][K|V][key][dim]
// for the tensor-core attention: dims (64 dims, page_size keys, head_dim / 64
// halves, layers x kv heads x 2 planes, n_pages), box 64 x att_box_keys x
// halves x 2 x 1 -- the K and V of 16 (or 64) keys of one (layer, kv head) in
// one copy, landing as [plane][half][key][64] -- 128-byte swizzle, zero fill
// outside.
int kv_make_map(CUtensorMap* map, const void* kv, int head_dim, int page_size, int planes, int n_pages,
                size_t page_elems);
// 3D byte tensor map over a stack of [rows][K] weight rows (esz bytes an
// element) for the streamed expert GEMVs: box 128 bytes x box_rows rows x
// box_chunks 128-byte chunks of K, landing as [chunk][row][128] with the
// 128-byte swizzle. Returns 0 on success.
int gemv_make_map(CUtensorMap* map, const void* base, int esz, uint64_t K, uint64_t rows, uint32_t box_rows,
                  uint32_t box_chunks);
// Keys per KV box of the tensor-core attention: a whole 64-key chunk when
// pages hold whole chunks (page_size a multiple of 64), else 16.
inline int att_box_keys(const Dims& D) { return D.P % 64 == 0 ? 64 : 16; }
// Rewrites W [rows, K] (row-major; bf16, or e4m3 when f8) into the tiled
// layout the tensor-core GEMM streams (rows a multiple of 128, K of 64).
int tc_pack_weights(void* dst, const void* src, int rows, int K, int f8, cudaStream_t st);
void launch_tc_gemm(const TcMaps& maps, const TcParams& P, int m_tiles, int groups, int n_tiles, cudaStream_t st);
// True when a bf16 single-operand launch of up to `rows` activation rows per
// CTA (two parts) takes the shared-memory column scan TC_ARGMAX / TC_STATS use.
bool tc_column_scan_fits(int rows);
cudaError_t configure_tc_kernels();
// out_lo2 (nullable): the third part bf16(v - hi - lo).
void launch_norm_bf16(const Dims& D, const float* x, const float* gamma, uint16_t* out, uint16_t* out_lo,
                      uint16_t* out_lo2, int T, int f16, cudaStream_t st);
void launch_rope_kv(const Dims& D, const DevState& S, const StepBuf& B, int layer, int T, cudaStream_t st);
void launch_gather_bf16(const Dims& D, const StepBuf& B, int T, cudaStream_t st);
void launch_argmax_commit(const Dims& D, const DevState& S, const StepBuf& B, int T, int ld, bool commit, int n_seq,
                          int K, cudaStream_t st);

// Kernel classes (for profiling); order matches spec_kernel_class_name().
enum KClass { KC_ASSEMBLE, KC_QKV, KC_ATTN, KC_OPROJ, KC_ROUTER, KC_GATEUP, KC_DOWN, KC_COMBINE, KC_LMHEAD,
              KC_COMMIT, KC_STAGE, KC_COUNT };
void launch_commit(const Dims& D, const DevState& S, const StepBuf& B, int n_seq, int K, cudaStream_t st);
// Commit of a sampled step from the sampler's [n_seq] accepted counts and tokens.
void launch_commit_sampled(const Dims& D, const DevState& S, const StepBuf& B, int n_seq, int K, const int* acc,
                           const int* tok, cudaStream_t st);
// Rejection sampling, cooperative form (ops_sample.cu): logits [n_seq][K+1][vocab];
// n_draft (nullable) gives each sequence's draft count (bonus row n_draft);
// 1 / temperature from it_dev when non-null, else `it`. ws: rs_coop_ws_bytes
// zero-filled bytes, left zeroed.
size_t rs_coop_ws_bytes(int n_seq, int K);
int rs_coop_blocks();   // blocks resident at once (queried once per device; 0 on failure)
cudaError_t launch_rs_coop(const float* logits, const int32_t* drafts, const int32_t* n_draft, const float* q,
                           const float* u_accept, const float* u_sample, int n_seq, int K, int vocab, float it,
                           const float* it_dev, int32_t* out_acc, int32_t* out_tok, void* ws, cudaStream_t st);
// Rejection sampling of a sampled step from the LM head's TC_STATS output
// (stats [rows][V / 128][4], xd [rows]), recomputing the picked tile's logits
// from the tiled bf16 LM head and the rows' hi / lo LM-head inputs; one block
// per sequence. Writes the sampler's [n_seq] accepted counts and tokens.
int rs_tiles_max_h();   // the widest LM-head input launch_rs_tiles takes
void launch_rs_tiles(const float* stats, const float* xd, int V, const uint16_t* lm_head_tiled, const uint16_t* xn_hi,
                     const uint16_t* xn_lo, int h, const int32_t* drafts, const int32_t* n_draft, const float* u_accept,
                     const float* u_sample, const float* it_dev, int n_seq, int K, int32_t* out_acc, int32_t* out_tok,
                     cudaStream_t st);
// [u_accept (max_batch K) | u_sample (max_batch (K+1)) | 1 / temperature] <- a sampled step's inputs.
void launch_stage_sample(float* dst, int max_batch, int K, const float* ua, const float* us, int n_seq, float it,
                         cudaStream_t st);
void launch_stage_dev(const StepBuf& B, int n_seq, int K, const int* seq_ids, const int* drafts,
                      const int* n_draft, int* out_acc, int* out_bonus, cudaStream_t st);
int launches_per_step(const Dims& D, int T);
// FastMTP draft-block input rows (ops_mtp.cu): cat = [N_e(E tok) ; N_h(N_o src)],
// z = P cat for n_rows rows (src[r] null: a padding row; tok[r] = -(j + 1):
// the token is drafts[j]).
void launch_mtp_input(const Dims& D, const int* tok, const float* const* src, const int* drafts, int n_rows,
                      const void* tok_embed,
                      const float* enorm, const float* final_norm, const float* hnorm, const void* P, float* cat,
                      float* z, cudaStream_t st);
// Record `msg` as the calling thread's last error (spec_last_error) and return code.
int set_last_error(int code, const char* msg);
// Programmatic dependent launch is used for every step kernel unless this
// thread turns it off (the profiler does, so its events bracket one kernel).
inline bool& pdl_enabled() {
  static thread_local bool on = true;
  return on;
}

template <class... KArgs, class... Args>
inline cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                            Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Opt a kernel in to the largest dynamic shared memory the device allows
// next to its static shared memory (an upper bound: occupancy follows the
// bytes each launch asks for). Called at model set-up, never during capture.
template <class K>
inline cudaError_t allow_dyn_smem(K kernel) {
  int dev = 0, optin = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  cudaFuncAttributes fa;
  if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, kernel);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, optin - (int)fa.sharedSizeBytes);
  return e;
}
cudaError_t configure_gemv_kernels();
cudaError_t configure_stream_kernels();
cudaError_t configure_attn_kernels();
cudaError_t configure_small_kernels();

}  // namespace spec
