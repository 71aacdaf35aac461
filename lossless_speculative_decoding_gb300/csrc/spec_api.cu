// C-ABI runtime of the verify-step library: model state, weight upload,
// prefill, verify steps (replayed as CUDA graphs per batch size), sequence
// and prefix management over the paged KV pool.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <atomic>
#include <chrono>
#include <cstdio>
#include <thread>
#include <cstring>
#include <map>
#include <memory>
#include <string>
#include <vector>

#include "../../include/spec.h"
#include "kernels.h"
#include "kv_pool.h"

using namespace spec;

namespace {

thread_local std::string g_last_error;

int fail(int code, const std::string& msg) {
  g_last_error = msg;
  return code;
}

#define CU(call)                                                                   \
  do {                                                                             \
    cudaError_t e_ = (call);                                                       \
    if (e_ != cudaSuccess)                                                         \
      return fail(SPEC_ERR_CUDA, std::string(#call) + ": " + cudaGetErrorString(e_)); \
  } while (0)

constexpr int PER_LAYER = 13;
constexpr int N_GLOBAL = 3;
constexpr int MAX_PREFIXES = 16;

int elt_bytes(int dtype) { return dtype == SPEC_F32 ? 4 : dtype == SPEC_BF16 ? 2 : 1; }

// (bytes) of tensor `idx` for `c`; -1 for a bad index.
int64_t tensor_bytes(const spec_config& c, int idx) {
  const int64_t h = c.hidden, d = c.head_dim, V = c.vocab;
  const int side = c.wdtype == SPEC_F32 ? SPEC_F32 : SPEC_BF16;
  const bool fp8 = c.wdtype == SPEC_FP8, q4 = c.wdtype == SPEC_NVFP4;
  const int64_t F = c.n_experts + c.n_shared, qkv = (int64_t)(c.n_q_heads + 2 * c.n_kv_heads) * d;
  if (idx < 0 || idx >= N_GLOBAL + PER_LAYER * c.n_layers) return -1;
  if (idx == 0 || idx == 2) return V * h * elt_bytes(side);
  if (idx == 1) return h * 4;
  const int j = (idx - N_GLOBAL) % PER_LAYER;
  // a matrix of `rows` x `cols` elements: nvfp4 records hold codes (1/2 byte)
  // and block scales (1/16 byte) per element
  auto mat = [&](int64_t rows, int64_t cols) { return q4 ? rows * cols / 2 + rows * cols / 16 : rows * cols * elt_bytes(c.wdtype); };
  auto scl = [&](int64_t fp8_n, int64_t q4_n) { return fp8 ? fp8_n * 4 : q4 ? q4_n * 4 : 0; };
  switch (j) {
    case 0: return h * 4;
    case 1: return mat(qkv, h);
    case 2: return scl(qkv, 1);
    case 3: return mat(h, (int64_t)c.n_q_heads * d);
    case 4: return scl(h, 1);
    case 5: return h * 4;
    case 6: return (int64_t)c.n_experts * h * elt_bytes(side);
    case 7: return F * mat(c.inter, h);
    case 8: return scl(F * c.inter, F);
    case 9: return F * mat(c.inter, h);
    case 10: return scl(F * c.inter, F);
    case 11: return F * mat(h, c.inter);
    case 12: return scl(F * h, F);
  }
  return -1;
}

int check_config(const spec_config& c) {
  if (c.n_layers < 1 || c.hidden < 64 || c.n_q_heads < 1 || c.n_kv_heads < 1 || c.vocab < 4)
    return fail(SPEC_ERR_ARG, "config: non-positive shape");
  if (c.head_dim != 64 && c.head_dim != 128) return fail(SPEC_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
  if (c.n_q_heads % c.n_kv_heads) return fail(SPEC_ERR_ARG, "n_q_heads must be a multiple of n_kv_heads");
  if (c.wdtype < SPEC_F32 || c.wdtype > SPEC_NVFP4) return fail(SPEC_ERR_ARG, "wdtype");
  if (c.wdtype == SPEC_NVFP4) {
    // the nvfp4 kernels are the <= 8-row GEMVs: 128-element steps, 16-row units
    if (c.max_batch * (c.max_draft + 1) > 8)
      return fail(SPEC_ERR_UNSUPPORTED, "nvfp4 weights: at most 8 rows per verify step");
    if (c.hidden % 128 || c.inter % 128 || (c.n_q_heads * c.head_dim) % 128 || c.vocab % 16)
      return fail(SPEC_ERR_UNSUPPORTED, "nvfp4 weights: hidden, inter and Hq * head_dim must be multiples of 128");
  }
  if (c.n_experts < 0 || c.top_k < 0 || c.n_shared < 0 || c.inter < 4) return fail(SPEC_ERR_ARG, "ffn shape");
  if (c.n_experts > 0 && (c.top_k < 1 || c.top_k > c.n_experts || c.top_k > 16))
    return fail(SPEC_ERR_ARG, "top_k must be in [1, min(n_experts, 16)]");
  if (c.n_experts > 256) return fail(SPEC_ERR_UNSUPPORTED, "at most 256 routed experts");
  if (c.n_experts > 0 && c.hidden * elt_bytes(c.wdtype == SPEC_F32 ? SPEC_F32 : SPEC_BF16) > 32 * 8 * 16)
    return fail(SPEC_ERR_UNSUPPORTED, "router rows above 4 KiB");
  if (c.n_experts == 0 && (c.n_shared != 1 || c.top_k != 0))
    return fail(SPEC_ERR_ARG, "a dense FFN is one shared expert with top_k = 0");
  if (c.n_experts + c.n_shared < 1) return fail(SPEC_ERR_ARG, "no FFN experts");
  if (c.page_size < 16 || c.page_size % 16) return fail(SPEC_ERR_ARG, "page_size must be a multiple of 16");
  if (c.max_draft < 0 || c.max_draft > 31) return fail(SPEC_ERR_ARG, "max_draft must be in [0, 31]");
  if (c.max_seqs < 1 || c.max_batch < 1 || c.max_batch > c.max_seqs) return fail(SPEC_ERR_ARG, "max_seqs/max_batch");
  if (c.max_ctx < c.max_draft + 2) return fail(SPEC_ERR_ARG, "max_ctx too small");
  if (c.n_pages < 1) return fail(SPEC_ERR_ARG, "n_pages");
  const int w = c.wdtype == SPEC_NVFP4 ? 1 : elt_bytes(c.wdtype);
  // 16-byte vector loads along every reduction dimension
  if ((c.hidden * w) % 16 || (c.inter * w) % 16 || (c.n_q_heads * c.head_dim * w) % 16 ||
      (c.hidden * elt_bytes(c.wdtype == SPEC_F32 ? SPEC_F32 : SPEC_BF16)) % 16)
    return fail(SPEC_ERR_UNSUPPORTED, "reduction dims must be multiples of 16 bytes");
  if (c.hidden % 4 || c.inter % 4 || c.vocab % 4) return fail(SPEC_ERR_UNSUPPORTED, "dims must be multiples of 4");
  return SPEC_OK;
}

struct Prefix {
  bool live = false;
  int slot = -1;                 // hidden pool slot holding the prefix pages
  std::vector<int32_t> tokens;
  int full_pages = 0;
};

// FastMTP draft head attached to a model ("Jina-OCR-v1", section 3.1). The
// shared draft block runs as an internal one-layer dense model `blk` whose
// sequence slot seq * Kmax + (k - 1) holds depth k's cache of sequence seq:
// row r of depth k sits at cache index r - (p0 + k - 1) and is rotated at
// absolute position r. Per call, every depth takes its newly committed rows
// (kept) and k - 1 speculative rows (recomputed by the next call), in passes
// of R rows (padding rows after the real ones).
struct MtpHead {
  spec_model* blk = nullptr;
  int Kmax = 0, R = 0, B0 = 0, ymax = 0;
  float* enorm = nullptr;
  float* hnorm = nullptr;
  void* P = nullptr;                    // eh_proj [h][2h]
  float* cat = nullptr;                 // [R][2h]
  float* Y = nullptr;                   // [Kmax][ymax][h] outputs (before N_o) of one call's rows, per depth
  float* ylast = nullptr;               // [max_seqs][Kmax][h] output of each depth's last committed row
  float* b0 = nullptr;                  // [max_seqs][B0][h] decoder states of prompt rows p0..
  int* d_meta = nullptr;                // one pass: [4][R] tokens, cache index, RoPE position, slot; [R] source rows
  int* d_drafts = nullptr;              // [Kmax] drafts of the call (tokens -(j + 1) read draft j)
  int pass_ints = 0, max_pass = 0;      // ints per pass (meta + pointers); passes per call
  int* pin = nullptr;                   // pinned staging: max_pass passes
  std::vector<int> p0, p_done, b0_rows, last_pos0, last_idx;
  std::vector<std::vector<int32_t>> prompt_tok;   // token id per prompt position (0 for visual rows)
  std::vector<void*> allocs;
  ~MtpHead() {
    if (blk) spec_free_model(blk);
    for (void* q : allocs) cudaFree(q);
    if (pin) cudaFreeHost(pin);
  }
};

}  // namespace

int spec::set_last_error(int code, const char* msg) { return fail(code, msg); }

// K splits of a tensor-core launch: when its CTAs (weight tiles x activation
// tiles x groups) leave SMs idle, as many splits as still fit in one wave of
// one CTA per SM, each keeping >= 16 K tiles and none empty. The CTA count is
// taken at the model's verify rows (max_batch x (K + 1)), a model constant,
// never at a step's own rows, so a row's arithmetic is the same in every
// step. MoE launches have many groups and never split.
static int tc_ksplit(int n_sm, int m_tiles, int groups, int n_tiles, int KT) {
  if (groups > 1) return 1;
  int ks = n_sm / (m_tiles * n_tiles);
  ks = std::min(ks, std::max(1, KT / 16));
  if (ks <= 1) return 1;
  const int kts = (KT + ks - 1) / ks;
  return (KT + kts - 1) / kts;
}

// activation rows per CTA of a dense tensor-core launch (see tc_dense); with
// three activation parts the MMA's N (3 x rows) stays within 256. A CTA's
// time is set by its K stream, not by its rows, so the launch takes the
// smallest tile whose CTAs fit in one wave (more CTAs only add waves), else
// the largest tile.
static int tc_dense_ntile(int n_sm, int M, int T, bool three_parts = false) {
  const int largest = three_parts ? 64 : 128;
  for (int nt = 32; nt < largest; nt *= 2)
    if ((M / 128) * ((T + nt - 1) / nt) <= n_sm) return nt;
  return largest;
}

struct spec_model {
  spec_config cfg{};
  cudaStream_t stream = nullptr;
  Dims D{};
  DevState S{};
  StepBuf B{};
  int K = 0, R = 1, Tmax = 1, prefill_chunk = 256;
  int Tv = 1;                      // verify rows of the largest batch (max_batch x R)
  std::vector<void*> allocs;
  std::vector<void*> wptr;         // device pointer per tensor (nullptr if absent)
  std::vector<LayerW> layers;
  std::vector<CUtensorMap> ffn_maps;       // [layer][gate, up, down] of the streamed expert GEMVs
  void* tok_embed = nullptr;
  void* lm_head = nullptr;
  float* final_norm = nullptr;
  std::unique_ptr<KvPool> pool;
  int n_slots = 0;                 // max_seqs + MAX_PREFIXES
  std::vector<char> busy;
  std::vector<int32_t> seq_len_h, last_tok_h, keep_h;
  std::vector<std::vector<int32_t>> gen;   // generated tokens (host view)
  std::vector<int32_t> bt_h;               // host copy of the device block tables
  std::vector<Prefix> prefixes;
  std::map<int, cudaGraphExec_t> graphs;
  int32_t* pin_in = nullptr;       // pinned staging (host)
  int32_t* pin_out = nullptr;
  int step_in_n = 0, step_out_n = 0;
  bool host_dirty = false;         // device state newer than host view (after _dev steps)
  bool own_stream = false;
  int64_t h2d_bytes = 0, d2h_bytes = 0;   // host<->device bytes moved by step calls
  std::atomic<int> prof_gate{1};           // profiler: stream held until a step is enqueued
  // tensor-core path (bf16 weights, more than 8 rows per step): tensor maps of
  // every weight and of the bf16 activation operands
  bool use_tc = false;
  float* tc_part = nullptr;                                     // split-K partials
  int* tc_cnt = nullptr;                                        // split-K tile arrival counters
  CUtensorMap kv_map{};                                        // paged KV pool (tensor-core attention)
  CUtensorMap tc_xn, tc_o, tc_xperm, tc_hperm;                 // activations: hi
  CUtensorMap tc_xn_lo, tc_o_lo, tc_xperm_lo, tc_hperm_lo;     //              lo
  CUtensorMap tc_xn_lo2;                                       //              lo2 (QKV input)

  MtpHead* mtp = nullptr;                 // draft head (spec_mtp_init), null without one

  // sampled steps (spec_verify_step_sample*), allocated on first use
  std::map<int, cudaGraphExec_t> graphs_sample;
  float* smp_logits = nullptr;     // [Tv][V] f32 logits of the step rows (no tile statistics)
  float* smp_stats = nullptr;      // [Tv][V / 128][4] LM-head tile statistics (tensor-core path)
  float* smp_xd = nullptr;         // [Tv] the rows' draft logits (tensor-core path)
  float* smp_in = nullptr;         // [u_accept (max_batch K) | u_sample (max_batch R) | 1 / temperature]
  int* smp_out = nullptr;          // [accepted (max_batch) | token (max_batch)] from the sampler
  void* smp_ws = nullptr;          // sampler workspace (zero-filled, left zeroed by every call)
  float* pin_smp = nullptr;        // pinned staging of smp_in (host-mode steps)

  ~spec_model() {
    delete mtp;
    for (auto& g : graphs) cudaGraphExecDestroy(g.second);
    for (auto& g : graphs_sample) cudaGraphExecDestroy(g.second);
    if (pin_smp) cudaFreeHost(pin_smp);
    if (own_stream) cudaStreamDestroy(stream);
    for (void* p : allocs) cudaFree(p);
    if (pin_in) cudaFreeHost(pin_in);
    if (pin_out) cudaFreeHost(pin_out);
  }

  template <class T>
  int dalloc(T** p, size_t n) {
    void* q = nullptr;
    if (n == 0) n = 1;
    cudaError_t e = cudaMalloc(&q, n * sizeof(T));
    if (e != cudaSuccess) return fail(SPEC_ERR_NOMEM, std::string("cudaMalloc: ") + cudaGetErrorString(e));
    allocs.push_back(q);
    *p = reinterpret_cast<T*>(q);
    return SPEC_OK;
  }

  int check_err() {
    int e = 0;
    CU(cudaMemcpyAsync(&e, S.err, sizeof(int), cudaMemcpyDeviceToHost, stream));
    CU(cudaStreamSynchronize(stream));
    if (e) {
      CU(cudaMemsetAsync(S.err, 0, sizeof(int), stream));
      return fail(SPEC_ERR_STATE, "device error bits " + std::to_string(e) +
                                       " (1 page, 2 token, 4 position out of range)");
    }
    return SPEC_OK;
  }

  // Upload block-table row of `slot` from the host allocator.
  int push_table(int slot) {
    const auto& t = pool->table(slot);
    int32_t* row = bt_h.data() + (size_t)slot * D.max_pages;
    std::fill(row, row + D.max_pages, -1);
    std::copy(t.begin(), t.end(), row);
    CU(cudaMemcpyAsync(const_cast<int*>(S.bt) + (size_t)slot * D.max_pages, row, D.max_pages * sizeof(int32_t),
                       cudaMemcpyHostToDevice, stream));
    h2d_bytes += (int64_t)D.max_pages * sizeof(int32_t);
    return SPEC_OK;
  }

  int push_seq_scalars(int slot) {
    CU(cudaMemcpyAsync(S.seq_len + slot, &seq_len_h[slot], 4, cudaMemcpyHostToDevice, stream));
    CU(cudaMemcpyAsync(S.last_tok + slot, &last_tok_h[slot], 4, cudaMemcpyHostToDevice, stream));
    CU(cudaMemcpyAsync(S.keep_pages + slot, &keep_h[slot], 4, cudaMemcpyHostToDevice, stream));
    return SPEC_OK;
  }

  // Profiling: events around every launch, active-expert counts per router.
  struct Prof {
    std::vector<cudaEvent_t> ev;
    std::vector<int> cls;
    int n = 0;
    int32_t* act = nullptr;      // pinned
    int nact = 0;
  };

  template <class F>
  void run_k(Prof* p, int cls, F&& launch) {
    if (p) cudaEventRecord(p->ev[2 * p->n], stream);
    launch();
    if (p) {
      cudaEventRecord(p->ev[2 * p->n + 1], stream);
      p->cls[p->n] = cls;
      p->n++;
    }
  }

  // Tensor-core GEMM launches. Dense: one group covering T rows. Grouped: the
  // active-expert list of the step (rows of the permuted operand).
  // blo2: a third activation part (the QKV input), else two parts
  void tc_dense(const void* w, const CUtensorMap& b, const CUtensorMap& blo, int K, int M, int T, int epi,
                float* out, int ldo, const float* scale = nullptr, const CUtensorMap* blo2 = nullptr,
                const StatsOut* stats = nullptr) {
    TcMaps mp;
    mp.b = b; mp.blo = blo; mp.blo2 = blo2 ? *blo2 : blo; mp.dual = 0; mp.f8 = scale != nullptr;
    TcParams P = {};
    P.wa = w; P.wa2 = w;
    P.K = K; P.Mg = M; P.N = T; P.ldo = ldo; P.epi = epi; P.out_f32 = out; P.err = S.err; P.split = blo2 ? 2 : 1;
    P.scale = scale;
    if (epi == TC_ARGMAX) { P.am_val = B.am_val; P.am_idx = B.am_idx; P.am_ld = M / 128; }
    if (epi == TC_STATS && stats) { P.st = *stats; P.am_ld = M / 128; }
    // too few CTAs for the GPU with 128-row activation tiles (small projections
    // at moderate T): 32-row tiles quadruple them; the weight tile is then read
    // by CTAs that run side by side (N tiles vary fastest) and hits in L2
    P.ntile = tc_dense_ntile(D.n_sm, M, T, blo2 != nullptr);
    const int tv = Tv, ntv = tc_dense_ntile(D.n_sm, M, tv, blo2 != nullptr);
    P.ksplit = tc_ksplit(D.n_sm, M / 128, 1, (tv + ntv - 1) / ntv, K / 64);
    P.part = tc_part; P.part_n = T; P.part_m = M; P.tile_cnt = tc_cnt;
    launch_tc_gemm(mp, P, M / 128, P.ksplit, (T + P.ntile - 1) / P.ntile, stream);
  }
  void tc_grouped(const void* w, const void* w2, const CUtensorMap& b, const CUtensorMap& blo, int K, int Mg, int T,
                  int epi, float* out_f32, uint16_t* out_bf16, uint16_t* out_lo, int ldo,
                  const float* scale = nullptr, const float* scale2 = nullptr) {
    TcMaps mp;
    mp.b = b; mp.blo = blo; mp.blo2 = blo; mp.dual = w2 ? 1 : 0; mp.f8 = scale != nullptr;
    TcParams P = {};
    P.wa = w; P.wa2 = w2 ? w2 : w;
    P.K = K; P.Mg = Mg; P.N = T; P.ldo = ldo; P.epi = epi; P.out_f32 = out_f32; P.out_bf16 = out_bf16;
    P.out_bf16_lo = out_lo; P.split = 1; P.scale = scale; P.scale2 = scale2;
    P.perm = B.perm; P.err = S.err;
    P.g_expert = B.act_expert; P.g_off = B.act_off; P.g_cnt = B.act_cnt; P.g_n = B.n_active;
    const int max_active = (D.E > 0 ? std::min(D.E, T * D.k) : 0) + D.S;
    P.ntile = 128;   // a small group's CTA still runs N = 32 with a deeper pipeline
    P.ksplit = tc_ksplit(D.n_sm, Mg / 128, max_active, (Tv * D.NS + 127) / 128, K / 64);
    P.part = tc_part; P.part_n = T * D.NS; P.part_m = Mg * max_active; P.tile_cnt = tc_cnt;
    launch_tc_gemm(mp, P, Mg / 128, max_active * P.ksplit, (T + 127) / 128, stream);
  }

  // Enqueue one forward over T rows already assembled in B (row meta + x);
  // returns the residual buffer holding the final rows.
  const float* enqueue_layers(int T, int R_rows, Prof* p = nullptr) {
    float* cur = B.x;
    const int qkv_rows = (D.Hq + 2 * D.Hkv) * D.d;
    for (int l = 0; l < D.L; ++l) {
      const LayerW& W = layers[l];
      if (use_tc) {
        run_k(p, KC_QKV, [&] {
          launch_norm_bf16(D, cur, W.attn_norm, B.xn_bf16, B.xn_lo, B.xn_lo2, T, D.op_f16, stream);
          tc_dense(W.w_qkv, tc_xn, tc_xn_lo, D.h, qkv_rows, T, TC_STORE, B.qkv, qkv_rows, W.s_qkv, &tc_xn_lo2);
          launch_rope_kv(D, S, B, l, T, stream);
        });
        run_k(p, KC_ATTN, [&] { launch_attn_part(D, S, B, l, T, R_rows, kv_map, stream); });
        run_k(p, KC_OPROJ, [&] { tc_dense(W.w_o, tc_o, tc_o_lo, D.Hq * D.d, D.h, T, TC_ADD, cur, D.h, W.s_o); });
        run_k(p, KC_ROUTER, [&] {
          launch_router(D, B, W, T, cur, true, stream);
          launch_gather_bf16(D, B, T, stream);
        });
        run_k(p, KC_GATEUP, [&] {
          tc_grouped(W.w_gate, W.w_up, tc_xperm, tc_xperm_lo, D.h, D.inter, T, TC_SWIGLU, nullptr, B.hperm,
                     B.hperm_lo, D.inter, W.s_gate, W.s_up);
        });
        if (p) cudaMemcpyAsync(p->act + p->nact++, B.n_active, 4, cudaMemcpyDeviceToHost, stream);
        run_k(p, KC_DOWN, [&] {
          tc_grouped(W.w_down, nullptr, tc_hperm, tc_hperm_lo, D.inter, D.h, T, TC_SCATTER, B.y, nullptr, nullptr,
                     D.h, W.s_down);
        });
        run_k(p, KC_COMBINE, [&] { launch_combine(D, B, cur, T, stream); });
        continue;
      }
      run_k(p, KC_QKV, [&] { launch_qkv(D, S, B, W, l, T, cur, stream); });
      run_k(p, KC_ATTN, [&] { launch_attn_part(D, S, B, l, T, R_rows, kv_map, stream); });
      run_k(p, KC_OPROJ, [&] { launch_oproj(D, B, W, T, cur, stream); });
      run_k(p, KC_ROUTER, [&] { launch_router(D, B, W, T, cur, false, stream); });
      run_k(p, KC_GATEUP, [&] { launch_gateup(D, B, W, T, S.err, stream); });
      if (p) cudaMemcpyAsync(p->act + p->nact++, B.n_active, 4, cudaMemcpyDeviceToHost, stream);
      run_k(p, KC_DOWN, [&] { launch_down(D, B, W, T, S.err, stream); });
      run_k(p, KC_COMBINE, [&] { launch_combine(D, B, cur, T, stream); });
    }
    return cur;
  }

  // Final norm + LM head + argmax over rows [0, T) of x (+ commit).
  void enqueue_lmhead(const float* x, int T, float* logits_dbg, bool commit, int n_seq) {
    if (!use_tc) {
      launch_lmhead_step(D, S, B, lm_head, final_norm, x, T, logits_dbg, commit, n_seq, K, stream);
      return;
    }
    launch_norm_bf16(D, x, final_norm, B.xn_bf16, B.xn_lo, nullptr, T, 0, stream);
    if (logits_dbg) tc_dense(lm_head, tc_xn, tc_xn_lo, D.h, D.V, T, TC_STORE, logits_dbg, D.V);
    tc_dense(lm_head, tc_xn, tc_xn_lo, D.h, D.V, T, TC_ARGMAX, nullptr, 0);
    launch_argmax_commit(D, S, B, T, D.V / 128, commit, n_seq, K, stream);
  }

  // Sampled step tail: the step rows' logits, rejection sampling over them
  // (drafts and draft counts from the staging block, uniforms and 1 /
  // temperature from smp_in), then the commit of what it decided.
  void enqueue_sample(const float* x, int T, int n_seq, Prof* p, cudaError_t* err) {
    const int mb = B.max_batch;
    if (smp_stats) {
      // tensor-core LM head: softmax statistics per 128-token tile instead of logits
      run_k(p, KC_LMHEAD, [&] {
        launch_norm_bf16(D, x, final_norm, B.xn_bf16, B.xn_lo, nullptr, T, 0, stream);
        StatsOut so{};
        so.out = smp_stats;
        so.xd = smp_xd;
        so.it = smp_in + mb * K + mb * R;
        so.drafts = B.step_in + mb;
        so.nd = B.step_in + mb + mb * K;
        so.K = K;
        so.R = R;
        tc_dense(lm_head, tc_xn, tc_xn_lo, D.h, D.V, T, TC_STATS, nullptr, 0, nullptr, nullptr, &so);
      });
      run_k(p, KC_COMMIT, [&] {
        launch_rs_tiles(smp_stats, smp_xd, D.V, static_cast<const uint16_t*>(lm_head), B.xn_bf16, B.xn_lo, D.h,
                        B.step_in + mb, B.step_in + mb + mb * K, smp_in, smp_in + mb * K, smp_in + mb * K + mb * R,
                        n_seq, K, smp_out, smp_out + mb, stream);
        launch_commit_sampled(D, S, B, n_seq, K, smp_out, smp_out + mb, stream);
      });
      return;
    }
    run_k(p, KC_LMHEAD, [&] {
      if (!use_tc) {
        launch_lmhead_step(D, S, B, lm_head, final_norm, x, T, smp_logits, false, n_seq, K, stream);
      } else {
        launch_norm_bf16(D, x, final_norm, B.xn_bf16, B.xn_lo, nullptr, T, 0, stream);
        tc_dense(lm_head, tc_xn, tc_xn_lo, D.h, D.V, T, TC_STORE, smp_logits, D.V);
      }
    });
    run_k(p, KC_COMMIT, [&] {
      const cudaError_t e = launch_rs_coop(smp_logits, B.step_in + mb, B.step_in + mb + mb * K, nullptr, smp_in,
                                           smp_in + mb * K, n_seq, K, D.V, 1.f, smp_in + mb * K + mb * R,
                                           smp_out, smp_out + mb, smp_ws, stream);
      if (e != cudaSuccess && err) *err = e;
      launch_commit_sampled(D, S, B, n_seq, K, smp_out, smp_out + mb, stream);
    });
  }

  void enqueue_verify(int n_seq, float* logits_dbg, bool commit, Prof* p = nullptr, bool sample = false,
                      cudaError_t* err = nullptr) {
    const int T = n_seq * R;
    run_k(p, KC_ASSEMBLE, [&] { launch_assemble_verify(D, S, B, tok_embed, n_seq, K, stream); });
    const float* xf = enqueue_layers(T, R, p);
    if (sample) {
      enqueue_sample(xf, T, n_seq, p, err);
      return;
    }
    run_k(p, KC_LMHEAD, [&] { enqueue_lmhead(xf, T, logits_dbg, commit, n_seq); });
  }

  // Buffers of the sampled steps, on first use.
  int ensure_sampling() {
    if (smp_logits || smp_stats) return SPEC_OK;
    if (D.V % 4 || D.V > 262144) return fail(SPEC_ERR_UNSUPPORTED, "sampled steps need vocab % 4 == 0 and <= 262144");
    if (rs_coop_blocks() < 1) return fail(SPEC_ERR_CUDA, "cannot size the sampler's cooperative launch");
    const int mb = B.max_batch;
    const size_t nin = (size_t)mb * K + (size_t)mb * R + 1;
    const size_t ws = rs_coop_ws_bytes(mb, K);
    int rc;
    char* w = nullptr;
    if ((rc = dalloc(&smp_in, nin)) || (rc = dalloc(&smp_out, 2 * (size_t)mb)) || (rc = dalloc(&w, ws))) return rc;
    CU(cudaMemsetAsync(w, 0, ws, stream));
    CU(cudaMallocHost(&pin_smp, nin * sizeof(float)));
    smp_ws = w;
    if (use_tc && D.V % 128 == 0 && D.h % 8 == 0 && D.h <= rs_tiles_max_h() && tc_column_scan_fits(std::min(Tv, 128)))
      return (rc = dalloc(&smp_xd, (size_t)Tv)) ? rc : dalloc(&smp_stats, (size_t)Tv * (D.V / 128) * 4);
    return dalloc(&smp_logits, (size_t)Tv * D.V);
  }

  int graph_for(int n_seq, cudaGraphExec_t* out, bool sample = false) {
    auto& cache = sample ? graphs_sample : graphs;
    auto it = cache.find(n_seq);
    if (it != cache.end()) { *out = it->second; return SPEC_OK; }
    cudaGraph_t g;
    CU(cudaStreamBeginCapture(stream, cudaStreamCaptureModeThreadLocal));
    cudaError_t le = cudaSuccess;
    enqueue_verify(n_seq, nullptr, true, nullptr, sample, &le);
    cudaError_t e = cudaStreamEndCapture(stream, &g);
    if (e == cudaSuccess && le != cudaSuccess) {
      cudaGraphDestroy(g);
      return fail(SPEC_ERR_CUDA, std::string("sampler launch: ") + cudaGetErrorString(le));
    }
    if (e != cudaSuccess) return fail(SPEC_ERR_CUDA, std::string("graph capture: ") + cudaGetErrorString(e));
    cudaGraphExec_t ge;
    e = cudaGraphInstantiate(&ge, g, 0);
    cudaGraphDestroy(g);
    if (e != cudaSuccess) return fail(SPEC_ERR_CUDA, std::string("graph instantiate: ") + cudaGetErrorString(e));
    cache[n_seq] = ge;
    *out = ge;
    return SPEC_OK;
  }

  bool seq_ok(int s) const { return s >= 0 && s < cfg.max_seqs && busy[s]; }
};

// The decoder's step buffer now holds other rows: no sequence can be drafted
// from the last step's states any more.
static void mtp_forget_steps(spec_model* m) {
  if (m->mtp) std::fill(m->mtp->last_idx.begin(), m->mtp->last_idx.end(), -1);
}

// ---------------------------------------------------------------------------
extern "C" {

const char* spec_strerror(int code) {
  switch (code) {
    case SPEC_OK: return "ok";
    case SPEC_ERR_ARG: return "invalid argument";
    case SPEC_ERR_NO_PAGES: return "KV page pool exhausted";
    case SPEC_ERR_CUDA: return "CUDA error";
    case SPEC_ERR_STATE: return "invalid state";
    case SPEC_ERR_NOMEM: return "out of memory";
    case SPEC_ERR_UNSUPPORTED: return "unsupported configuration";
  }
  return "unknown error";
}

const char* spec_last_error(void) { return g_last_error.c_str(); }

int spec_tensor_count(const spec_config* cfg) {
  if (!cfg || cfg->n_layers < 1) return fail(SPEC_ERR_ARG, "config");
  return N_GLOBAL + PER_LAYER * cfg->n_layers;
}

int64_t spec_tensor_bytes(const spec_config* cfg, int index) {
  if (!cfg) return fail(SPEC_ERR_ARG, "config");
  const int64_t b = tensor_bytes(*cfg, index);
  return b < 0 ? fail(SPEC_ERR_ARG, "tensor index") : b;
}

int spec_init_model(const spec_config* cfg_in, const void* const* host_tensors, uintptr_t cuda_stream,
                     spec_model** out_model) {
  if (!cfg_in || !out_model || !host_tensors) return fail(SPEC_ERR_ARG, "null argument");
  *out_model = nullptr;
  int rc = check_config(*cfg_in);
  if (rc) return rc;
  std::unique_ptr<spec_model> m(new spec_model());
  spec_config& c = m->cfg;
  c = *cfg_in;
  m->stream = reinterpret_cast<cudaStream_t>(cuda_stream);
  if (m->stream == nullptr) {   // the legacy default stream cannot be captured into a graph
    CU(cudaStreamCreateWithFlags(&m->stream, cudaStreamNonBlocking));
    m->own_stream = true;
  }
  m->K = c.max_draft;
  m->R = c.max_draft + 1;
  m->prefill_chunk = c.prefill_chunk > 0 ? c.prefill_chunk : 256;
  m->Tmax = std::max(c.max_batch * m->R, m->prefill_chunk);
  m->Tv = c.max_batch * m->R;
  Dims& D = m->D;
  D.L = c.n_layers; D.h = c.hidden; D.Hq = c.n_q_heads; D.Hkv = c.n_kv_heads; D.d = c.head_dim;
  D.E = c.n_experts; D.k = c.top_k; D.S = c.n_shared; D.inter = c.inter; D.V = c.vocab;
  D.wdtype = c.wdtype; D.act_f32 = c.wdtype == SPEC_F32; D.P = c.page_size;
  D.max_ctx = c.max_ctx; D.NS = c.top_k + c.n_shared; D.eps = c.rms_eps; D.theta = c.rope_theta;
  D.max_pages = (c.max_ctx + c.page_size - 1) / c.page_size;
  {
    int dev = 0;
    CU(cudaGetDevice(&dev));
    CU(cudaDeviceGetAttribute(&D.n_sm, cudaDevAttrMultiProcessorCount, dev));
  }
  D.page_elems = (size_t)c.n_layers * 2 * c.n_kv_heads * c.page_size * c.head_dim;
  if (attn_groups(D, c.max_batch * m->R, m->R) > ATT_MAX_GROUPS ||
      attn_groups(D, m->prefill_chunk, m->prefill_chunk) > ATT_MAX_GROUPS)
    return fail(SPEC_ERR_ARG, "max_batch x ceil((max_draft + 1) / rows per group) exceeds the attention group limit");
  const size_t kv_elt = D.act_f32 ? 4 : 2;

  CU(configure_gemv_kernels());
  CU(configure_stream_kernels());
  CU(configure_attn_kernels());
  CU(configure_small_kernels());

  // ---- weights ----
  const int nt = N_GLOBAL + PER_LAYER * c.n_layers;
  m->wptr.assign(nt, nullptr);
  for (int i = 0; i < nt; ++i) {
    const int64_t nb = tensor_bytes(c, i);
    if (nb == 0) continue;
    if (!host_tensors[i]) return fail(SPEC_ERR_ARG, "missing tensor " + std::to_string(i));
    char* p = nullptr;
    if ((rc = m->dalloc(&p, (size_t)nb))) return rc;
    CU(cudaMemcpy(p, host_tensors[i], (size_t)nb, cudaMemcpyHostToDevice));
    m->wptr[i] = p;
  }
  m->tok_embed = m->wptr[0];
  m->final_norm = (float*)m->wptr[1];
  m->lm_head = m->wptr[2];
  for (int l = 0; l < c.n_layers; ++l) {
    void** w = m->wptr.data() + N_GLOBAL + PER_LAYER * l;
    LayerW L;
    L.attn_norm = (const float*)w[0]; L.w_qkv = w[1]; L.s_qkv = (const float*)w[2];
    L.w_o = w[3]; L.s_o = (const float*)w[4]; L.ffn_norm = (const float*)w[5]; L.w_router = w[6];
    L.w_gate = w[7]; L.s_gate = (const float*)w[8]; L.w_up = w[9]; L.s_up = (const float*)w[10];
    L.w_down = w[11]; L.s_down = (const float*)w[12];
    L.ffn_map = nullptr; L.kst_gu = L.kst_dn = 0;
    m->layers.push_back(L);
  }

  // ---- KV pool and sequence state ----
  m->n_slots = c.max_seqs + MAX_PREFIXES;
  m->pool.reset(new KvPool(c.n_pages, c.page_size, m->n_slots, D.max_pages));
  if ((rc = m->dalloc((char**)&m->S.kv, (size_t)c.n_pages * D.page_elems * kv_elt))) return rc;
  if (!D.act_f32 && (D.d == 64 || D.d == 128) &&
      kv_make_map(&m->kv_map, m->S.kv, D.d, D.P, D.L * 2 * D.Hkv, c.n_pages, D.page_elems))
    return fail(SPEC_ERR_CUDA, "KV pool tensor map");
  int* bt = nullptr;
  if ((rc = m->dalloc(&bt, (size_t)m->n_slots * D.max_pages))) return rc;
  m->S.bt = bt;
  CU(cudaMemset(bt, 0xFF, (size_t)m->n_slots * D.max_pages * sizeof(int)));
  if ((rc = m->dalloc(&m->S.seq_len, m->n_slots))) return rc;
  if ((rc = m->dalloc(&m->S.last_tok, m->n_slots))) return rc;
  if ((rc = m->dalloc(&m->S.keep_pages, m->n_slots))) return rc;
  if ((rc = m->dalloc(&m->S.n_out, m->n_slots))) return rc;
  if ((rc = m->dalloc(&m->S.out_tok, (size_t)m->n_slots * c.max_ctx))) return rc;
  if ((rc = m->dalloc(&m->S.err, 1))) return rc;
  CU(cudaMemset(m->S.seq_len, 0, m->n_slots * 4));
  CU(cudaMemset(m->S.last_tok, 0, m->n_slots * 4));
  CU(cudaMemset(m->S.keep_pages, 0, m->n_slots * 4));
  CU(cudaMemset(m->S.n_out, 0, m->n_slots * 4));
  CU(cudaMemset(m->S.err, 0, 4));
  float *rc_cos = nullptr, *rc_sin = nullptr;
  if ((rc = m->dalloc(&rc_cos, (size_t)c.max_ctx * (c.head_dim / 2)))) return rc;
  if ((rc = m->dalloc(&rc_sin, (size_t)c.max_ctx * (c.head_dim / 2)))) return rc;
  m->S.rope_cos = rc_cos;
  m->S.rope_sin = rc_sin;
  launch_rope_table(D, rc_cos, rc_sin, m->stream);
  m->busy.assign(m->n_slots, 0);
  m->seq_len_h.assign(m->n_slots, 0);
  m->last_tok_h.assign(m->n_slots, 0);
  m->keep_h.assign(m->n_slots, 0);
  m->gen.assign(m->n_slots, {});
  m->bt_h.assign((size_t)m->n_slots * D.max_pages, -1);
  m->prefixes.assign(MAX_PREFIXES, Prefix());

  // ---- step buffers ----
  StepBuf& B = m->B;
  const int T = m->Tmax, NS = D.NS;
  B.n_chunk_max = (c.max_ctx + ATT_CHUNK - 1) / ATT_CHUNK;
  B.n_vblocks = lmhead_step_warps(D);             // one argmax candidate per LM-head warp
  B.max_batch = c.max_batch;
  const int max_active = (D.E > 0 ? std::min(D.E, T * std::max(D.k, 1)) : 0) + D.S;
  if ((rc = m->dalloc(&B.row_tok, T)) || (rc = m->dalloc(&B.row_pos, T)) || (rc = m->dalloc(&B.row_seq, T)) ||
      (rc = m->dalloc(&B.row_src, T)) || (rc = m->dalloc(&B.x, (size_t)T * D.h)) ||
      (rc = m->dalloc(&B.q, (size_t)T * D.Hq * D.d)) ||
      (rc = m->dalloc(&B.att_o, (size_t)T * D.Hq * B.n_chunk_max * D.d)) ||
      (rc = m->dalloc(&B.att_ml, (size_t)T * D.Hq * B.n_chunk_max * 2)) ||
      (rc = m->dalloc(&B.o, (size_t)T * D.Hq * D.d)) || (rc = m->dalloc(&B.u, (size_t)T * D.h)) ||
      (rc = m->dalloc(&B.ids, (size_t)T * std::max(D.k, 1))) ||
      (rc = m->dalloc(&B.wts, (size_t)T * std::max(D.k, 1))) || (rc = m->dalloc(&B.perm, (size_t)T * NS)) ||
      (rc = m->dalloc(&B.act_expert, max_active)) || (rc = m->dalloc(&B.act_off, max_active)) ||
      (rc = m->dalloc(&B.act_cnt, max_active)) || (rc = m->dalloc(&B.n_active, 1)) ||
      (rc = m->dalloc(&B.counter, 4)) || (rc = m->dalloc(&B.rlogit, (size_t)T * std::max(D.E, 1))) ||
      (rc = m->dalloc(&B.cnt_row, T)) || (rc = m->dalloc(&B.cnt_att, (size_t)T * D.Hkv)) ||
      (rc = m->dalloc(&B.cnt_lm, (T + GEMV_TP - 1) / GEMV_TP)) || (rc = m->dalloc(&B.h_act, (size_t)T * NS * D.inter)) ||
      (rc = m->dalloc(&B.y, (size_t)T * NS * D.h)) ||
      (rc = m->dalloc(&B.am_val, (size_t)T * B.n_vblocks)) || (rc = m->dalloc(&B.am_idx, (size_t)T * B.n_vblocks)) ||
      (rc = m->dalloc(&B.g, T)))
    return rc;
  // tensor-core path: bf16 or e4m3 weights with more than 8 rows per verify step
  {
    const int qkv_rows = (D.Hq + 2 * D.Hkv) * D.d;
    const bool shapes = D.h % 128 == 0 && qkv_rows % 128 == 0 && D.inter % 128 == 0 && D.V % 128 == 0 &&
                        (D.Hq * D.d) % 64 == 0 && D.h % 64 == 0 && D.inter % 64 == 0;
    m->use_tc = (c.wdtype == SPEC_BF16 || c.wdtype == SPEC_FP8) && c.max_batch * m->R > 8 && shapes;
    D.op_f16 = m->use_tc && c.wdtype == SPEC_FP8 ? 1 : 0;
  }
  if (!m->use_tc && (c.wdtype == SPEC_BF16 || c.wdtype == SPEC_FP8)) {
    // steps of at most 8 rows: the expert GEMVs stream their weights by TMA
    // when the shapes split into whole 128-byte chunks (else the register form)
    const int esz = c.wdtype == SPEC_BF16 ? 2 : 1;
    const int kgu = ffn_stage_k(D.h, esz), kdn = ffn_stage_k(D.inter, esz);
    if (kgu > 0 && kdn > 0 && D.inter % 8 == 0 && D.h % 16 == 0) {
      const int F = D.E + D.S;
      m->ffn_maps.resize((size_t)3 * D.L);
      for (int l = 0; l < D.L; ++l) {
        LayerW& W = m->layers[l];
        CUtensorMap* mp = m->ffn_maps.data() + 3 * l;
        if (gemv_make_map(mp, W.w_gate, esz, D.h, (uint64_t)F * D.inter, 8, kgu * esz / 128) ||
            gemv_make_map(mp + 1, W.w_up, esz, D.h, (uint64_t)F * D.inter, 8, kgu * esz / 128) ||
            gemv_make_map(mp + 2, W.w_down, esz, D.inter, (uint64_t)F * D.h, 16, kdn * esz / 128))
          return fail(SPEC_ERR_CUDA, "expert weight tensor maps");
        W.ffn_map = mp;
        W.kst_gu = kgu;
        W.kst_dn = kdn;
      }
    }
  }
  if (m->use_tc) {
    const int qkv_rows = (D.Hq + 2 * D.Hkv) * D.d;
    if ((rc = m->dalloc(&B.qkv, (size_t)T * qkv_rows)) || (rc = m->dalloc(&B.xn_bf16, (size_t)T * D.h)) ||
        (rc = m->dalloc(&B.xn_lo, (size_t)T * D.h)) || (rc = m->dalloc(&B.xn_lo2, (size_t)T * D.h)) ||
        (rc = m->dalloc(&B.o_bf16, (size_t)T * D.Hq * D.d)) ||
        (rc = m->dalloc(&B.o_lo, (size_t)T * D.Hq * D.d)) || (rc = m->dalloc(&B.xperm, (size_t)T * NS * D.h)) ||
        (rc = m->dalloc(&B.xperm_lo, (size_t)T * NS * D.h)) || (rc = m->dalloc(&B.hperm, (size_t)T * NS * D.inter)) ||
        (rc = m->dalloc(&B.hperm_lo, (size_t)T * NS * D.inter)))
      return rc;
    CU(configure_tc_kernels());
    const int F = D.E + D.S;
    // weights the tensor cores stream are rewritten, in place, into the tiled
    // layout (one contiguous swizzled block per 128 x 64 tile); the SIMT
    // kernels that read them row-major do not run on this path
    const int f8 = c.wdtype == SPEC_FP8 ? 1 : 0;
    struct Mat { void* p; int rows, K, f8; };
    std::vector<Mat> mats;
    for (int l = 0; l < D.L; ++l) {
      const LayerW& W = m->layers[l];
      mats.push_back({const_cast<void*>(W.w_qkv), qkv_rows, D.h, f8});
      mats.push_back({const_cast<void*>(W.w_o), D.h, D.Hq * D.d, f8});
      mats.push_back({const_cast<void*>(W.w_gate), F * D.inter, D.h, f8});
      mats.push_back({const_cast<void*>(W.w_up), F * D.inter, D.h, f8});
      mats.push_back({const_cast<void*>(W.w_down), F * D.h, D.inter, f8});
    }
    mats.push_back({m->lm_head, D.V, D.h, 0});
    size_t tmp_bytes = 0;
    for (const Mat& x : mats) tmp_bytes = std::max(tmp_bytes, (size_t)x.rows * x.K * (x.f8 ? 1 : 2));
    void* tmp = nullptr;
    CU(cudaMalloc(&tmp, tmp_bytes));
    int bad = 0;
    for (const Mat& x : mats) {
      const size_t nb = (size_t)x.rows * x.K * (x.f8 ? 1 : 2);
      bad |= tc_pack_weights(tmp, x.p, x.rows, x.K, x.f8, m->stream);
      if (cudaMemcpyAsync(x.p, tmp, nb, cudaMemcpyDeviceToDevice, m->stream) != cudaSuccess) bad = 1;
    }
    const cudaError_t se = cudaStreamSynchronize(m->stream);
    cudaFree(tmp);
    if (bad || se != cudaSuccess) return fail(SPEC_ERR_CUDA, "weight tiling failed");
    bad |= tc_make_map(&m->tc_xn, B.xn_bf16, D.h, T, 32);
    bad |= tc_make_map(&m->tc_o, B.o_bf16, (uint64_t)D.Hq * D.d, T, 32);
    bad |= tc_make_map(&m->tc_xperm, B.xperm, D.h, (uint64_t)T * NS, 32);
    bad |= tc_make_map(&m->tc_hperm, B.hperm, D.inter, (uint64_t)T * NS, 32);
    bad |= tc_make_map(&m->tc_xn_lo, B.xn_lo, D.h, T, 32);
    bad |= tc_make_map(&m->tc_xn_lo2, B.xn_lo2, D.h, T, 32);
    bad |= tc_make_map(&m->tc_o_lo, B.o_lo, (uint64_t)D.Hq * D.d, T, 32);
    bad |= tc_make_map(&m->tc_xperm_lo, B.xperm_lo, D.h, (uint64_t)T * NS, 32);
    bad |= tc_make_map(&m->tc_hperm_lo, B.hperm_lo, D.inter, (uint64_t)T * NS, 32);
    if (bad) return fail(SPEC_ERR_CUDA, "tensor map encoding failed");
    // split-K scratch: the largest [splits][1 + dual][rows][features] of the step's launches
    {
      const int tv = m->Tv;
      auto dn = [&](int M, bool three = false) {
        const int nt = tc_dense_ntile(D.n_sm, M, tv, three);
        return (tv + nt - 1) / nt;
      };
      const int ks_q = tc_ksplit(D.n_sm, qkv_rows / 128, 1, dn(qkv_rows, true), D.h / 64);
      const int ks_o = tc_ksplit(D.n_sm, D.h / 128, 1, dn(D.h), D.Hq * D.d / 64);
      const int ks_l = tc_ksplit(D.n_sm, D.V / 128, 1, dn(D.V), D.h / 64);
      const int gmin = (D.E > 0 ? 1 : 0) + D.S;        // fewest groups an expert launch can have
      const int ga = (D.E > 0 ? std::min(D.E, T * D.k) : 0) + D.S;   // most groups
      const int ks_g = tc_ksplit(D.n_sm, D.inter / 128, gmin, (tv * NS + 127) / 128, D.h / 64);
      const int ks_d = tc_ksplit(D.n_sm, D.h / 128, gmin, (tv * NS + 127) / 128, D.inter / 64);
      size_t part = 0, tiles = 0;
      auto need = [&](int ks, int dual, size_t rows, size_t feats, size_t mtiles, size_t ntiles) {
        if (ks <= 1) return;
        part = std::max(part, (size_t)ks * (1 + dual) * rows * feats);
        tiles = std::max(tiles, mtiles * ntiles);
      };
      need(ks_q, 0, T, qkv_rows, qkv_rows / 128, (T + 31) / 32);
      need(ks_o, 0, T, D.h, D.h / 128, (T + 31) / 32);
      need(ks_l, 0, T, D.V, D.V / 128, (T + 31) / 32);
      need(ks_g, 1, (size_t)T * NS, (size_t)D.inter * ga, D.inter / 128, ((size_t)T * NS + 127) / 128);
      need(ks_d, 0, (size_t)T * NS, (size_t)D.h * ga, D.h / 128, ((size_t)T * NS + 127) / 128);
      if (part) {
        if ((rc = m->dalloc(&m->tc_part, part)) || (rc = m->dalloc(&m->tc_cnt, tiles))) return rc;
        CU(cudaMemset(m->tc_cnt, 0, tiles * sizeof(int)));
      }
    }
  }
  m->step_in_n = c.max_batch * (2 + m->K);
  m->step_out_n = 2 * c.max_batch + 1;   // acc | bonus | device error bits
  // [out_ptrs (2 x 64-bit) | step inputs]: one host copy refreshes both
  int* stage = nullptr;
  if ((rc = m->dalloc(&stage, 4 + m->step_in_n)) || (rc = m->dalloc(&B.step_out, m->step_out_n))) return rc;
  B.out_ptrs = reinterpret_cast<unsigned long long*>(stage);
  B.step_in = stage + 4;
  CU(cudaMemset(B.counter, 0, 4 * sizeof(int)));
  CU(cudaMemset(B.cnt_row, 0, (size_t)T * sizeof(int)));
  CU(cudaMemset(B.cnt_att, 0, (size_t)T * D.Hkv * sizeof(int)));
  CU(cudaMemset(B.cnt_lm, 0, ((T + GEMV_TP - 1) / GEMV_TP) * sizeof(int)));
  CU(cudaMemset(stage, 0, (4 + m->step_in_n) * sizeof(int)));
  CU(cudaMallocHost(&m->pin_in, std::max(4 + m->step_in_n, T) * sizeof(int32_t)));
  CU(cudaMallocHost(&m->pin_out, std::max(m->step_out_n, T) * sizeof(int32_t)));
  CU(cudaStreamSynchronize(m->stream));
  CU(cudaGetLastError());
  *out_model = m.release();
  return SPEC_OK;
}

int spec_free_model(spec_model* m) {
  if (!m) return fail(SPEC_ERR_ARG, "null model");
  cudaStreamSynchronize(m->stream);
  delete m;
  return SPEC_OK;
}

// Run the prompt rows [start, start + n) of slot `slot` (rows described by
// `src`: token id >= 0 or -(visual row + 1)); returns the greedy token of the
// last row in *out_tok when out_tok != nullptr.
static int run_prefill_rows(spec_model* m, int slot, const std::vector<int32_t>& src, int start,
                            const void* vis, int32_t* out_tok) {
  const int n = (int)src.size();
  int first = -1;
  for (int c0 = 0; c0 < n; c0 += m->prefill_chunk) {
    const int T = std::min(m->prefill_chunk, n - c0);
    std::memcpy(m->pin_in, src.data() + c0, T * sizeof(int32_t));
    CU(cudaMemcpyAsync(m->B.row_src, m->pin_in, T * sizeof(int32_t), cudaMemcpyHostToDevice, m->stream));
    launch_assemble_prefill(m->D, m->S, m->B, m->tok_embed, vis, slot, start + c0, T, m->stream);
    const float* xf = m->enqueue_layers(T, T);
    if (m->mtp && slot < m->cfg.max_seqs && m->mtp->p0[slot] >= 0) {
      // the draft head's first call needs the decoder states of rows p0.. (kept while they fit)
      MtpHead& H = *m->mtp;
      const int a = std::max(H.p0[slot], start + c0), b = std::min(start + c0 + T, H.p0[slot] + H.B0);
      if (b > a)
        CU(cudaMemcpyAsync(H.b0 + ((size_t)slot * H.B0 + (a - H.p0[slot])) * m->D.h, xf + (size_t)(a - start - c0) * m->D.h,
                           (size_t)(b - a) * m->D.h * sizeof(float), cudaMemcpyDeviceToDevice, m->stream));
    }
    if (c0 + T == n && out_tok) {
      m->enqueue_lmhead(xf + (size_t)(T - 1) * m->D.h, 1, nullptr, false, 0);
      CU(cudaMemcpyAsync(m->pin_out, m->B.g, sizeof(int32_t), cudaMemcpyDeviceToHost, m->stream));
    }
    // the staging buffer is reused by the next chunk
    CU(cudaStreamSynchronize(m->stream));
    CU(cudaGetLastError());
    if (c0 + T == n && out_tok) first = m->pin_out[0];
  }
  int rc = m->check_err();
  if (rc) return rc;
  if (out_tok) *out_tok = first;
  return SPEC_OK;
}

int spec_register_prefix(spec_model* m, const int32_t* tok, int n_tok, int32_t* out_prefix_id) {
  if (!m || !tok || n_tok < 1 || !out_prefix_id) return fail(SPEC_ERR_ARG, "bad prefix arguments");
  for (int i = 0; i < n_tok; ++i)
    if (tok[i] < 0 || tok[i] >= m->cfg.vocab) return fail(SPEC_ERR_ARG, "prefix token out of range");
  if (n_tok + m->R + 1 > m->cfg.max_ctx) return fail(SPEC_ERR_ARG, "prefix longer than max_ctx");
  int id = -1;
  for (int i = 0; i < MAX_PREFIXES; ++i)
    if (!m->prefixes[i].live) { id = i; break; }
  if (id < 0) return fail(SPEC_ERR_STATE, "no free prefix slot");
  const int slot = m->cfg.max_seqs + id;
  int rc = m->pool->reserve(slot, n_tok);
  if (rc) return fail(rc, "prefix: KV pool exhausted");
  if ((rc = m->push_table(slot))) { m->pool->release(slot); return rc; }
  std::vector<int32_t> src(tok, tok + n_tok);
  mtp_forget_steps(m);
  rc = run_prefill_rows(m, slot, src, 0, nullptr, nullptr);
  if (rc) { m->pool->release(slot); m->push_table(slot); return rc; }
  Prefix& p = m->prefixes[id];
  p.live = true;
  p.slot = slot;
  p.tokens = src;
  p.full_pages = n_tok / m->cfg.page_size;
  // keep only the full pages: the partial tail is recomputed by each user
  m->pool->commit(slot, p.full_pages * m->cfg.page_size, 0);
  if ((rc = m->push_table(slot))) return rc;
  CU(cudaStreamSynchronize(m->stream));
  *out_prefix_id = id;
  return SPEC_OK;
}

int spec_release_prefix(spec_model* m, int32_t prefix_id) {
  if (!m || prefix_id < 0 || prefix_id >= MAX_PREFIXES || !m->prefixes[prefix_id].live)
    return fail(SPEC_ERR_ARG, "bad prefix id");
  Prefix& p = m->prefixes[prefix_id];
  m->pool->release(p.slot);
  int rc = m->push_table(p.slot);
  p = Prefix();
  CU(cudaStreamSynchronize(m->stream));
  return rc;
}

int spec_prefill(spec_model* m, int32_t seq_id, int32_t prefix_id, const void* vis_embeds_dev, int n_vis,
                 const int32_t* tok, int n_tok, int32_t* out_first_token) {
  if (!m || !out_first_token || n_vis < 0 || n_tok < 0 || (n_tok > 0 && !tok) || (n_vis > 0 && !vis_embeds_dev))
    return fail(SPEC_ERR_ARG, "bad prefill arguments");
  if (seq_id < 0 || seq_id >= m->cfg.max_seqs) return fail(SPEC_ERR_ARG, "seq_id out of range");
  if (m->busy[seq_id]) return fail(SPEC_ERR_STATE, "sequence slot busy");
  if (m->host_dirty) return fail(SPEC_ERR_STATE, "call spec_sync_seqs after device-resident steps");
  const Prefix* pre = nullptr;
  if (prefix_id >= 0) {
    if (prefix_id >= MAX_PREFIXES || !m->prefixes[prefix_id].live) return fail(SPEC_ERR_ARG, "bad prefix id");
    pre = &m->prefixes[prefix_id];
  }
  for (int i = 0; i < n_tok; ++i)
    if (tok[i] < 0 || tok[i] >= m->cfg.vocab) return fail(SPEC_ERR_ARG, "token out of range");
  const int n_pre = pre ? (int)pre->tokens.size() : 0;
  const int len = n_pre + n_vis + n_tok;
  if (len < 1) return fail(SPEC_ERR_ARG, "empty prompt");
  if (len + m->R > m->cfg.max_ctx) return fail(SPEC_ERR_ARG, "prompt + draft rows exceed max_ctx");
  KvPool& pool = *m->pool;
  int start = 0;
  if (pre && pre->full_pages > 0) {
    int rc = pool.share(pre->slot, pre->full_pages, seq_id);
    if (rc) return fail(rc, "prefix share failed");
    start = pre->full_pages * m->cfg.page_size;
  }
  int rc = pool.reserve(seq_id, len + m->R);
  if (rc) { pool.release(seq_id); return fail(rc, "KV pool exhausted"); }
  if ((rc = m->push_table(seq_id))) { pool.release(seq_id); return rc; }
  std::vector<int32_t> src;
  src.reserve(len - start);
  for (int p = start; p < len; ++p) {
    if (p < n_pre) src.push_back(pre->tokens[p]);
    else if (p < n_pre + n_vis) src.push_back(-(p - n_pre) - 1);
    else src.push_back(tok[p - n_pre - n_vis]);
  }
  if (m->mtp) {
    // the head's grid starts at the last visual row (row 0 without visual rows);
    // sequences with a shared prefix are not drafted by the head
    MtpHead& H = *m->mtp;
    H.p0[seq_id] = pre ? -1 : std::max(n_vis - 1, 0);
    H.p_done[seq_id] = H.p0[seq_id] - 1;
    H.b0_rows[seq_id] = std::max(0, std::min(H.B0, len - std::max(H.p0[seq_id], 0)));
    H.last_idx[seq_id] = -1;
    H.prompt_tok[seq_id].assign(len, 0);
    for (int i = 0; i < n_tok; ++i) H.prompt_tok[seq_id][n_pre + n_vis + i] = tok[i];
    for (int k = 0; k < H.Kmax; ++k) H.blk->pool->release(seq_id * H.Kmax + k);
  }
  int32_t first = -1;
  mtp_forget_steps(m);
  rc = run_prefill_rows(m, seq_id, src, start, vis_embeds_dev, &first);
  if (rc) { pool.release(seq_id); m->push_table(seq_id); return rc; }
  m->busy[seq_id] = 1;
  m->seq_len_h[seq_id] = len;
  m->last_tok_h[seq_id] = first;
  m->keep_h[seq_id] = 0;
  m->gen[seq_id].assign(1, first);
  pool.set_length(seq_id, len);
  int one = 1;
  if ((rc = m->push_seq_scalars(seq_id))) return rc;
  CU(cudaMemcpyAsync(m->S.out_tok + (size_t)seq_id * m->cfg.max_ctx, &first, 4, cudaMemcpyHostToDevice, m->stream));
  CU(cudaMemcpyAsync(m->S.n_out + seq_id, &one, 4, cudaMemcpyHostToDevice, m->stream));
  CU(cudaStreamSynchronize(m->stream));
  *out_first_token = first;
  return SPEC_OK;
}

// Inputs of a sampled step (host arrays).
struct SampleArgs {
  const float* u_accept;   // [n_seq][K]
  const float* u_sample;   // [n_seq][K+1]
  float temperature;
};

// Host-mode step common to spec_verify_step(_batch), spec_verify_step_sample_batch
// and spec_debug_logits.
static int verify_host(spec_model* m, int n_seq, const int32_t* seq_ids, const int32_t* drafts,
                       const int32_t* n_draft, int32_t* out_acc, int32_t* out_bonus, float* logits_dev,
                       const SampleArgs* smp = nullptr) {
  if (!m || n_seq < 1 || n_seq > m->cfg.max_batch || !seq_ids) return fail(SPEC_ERR_ARG, "bad batch");
  if (m->K > 0 && !drafts) return fail(SPEC_ERR_ARG, "null drafts");
  if (smp) {
    if (!(smp->temperature > 0.f) || !std::isfinite(1.f / smp->temperature))
      return fail(SPEC_ERR_ARG, "temperature must be positive");
    if (!smp->u_sample || (m->K > 0 && !smp->u_accept)) return fail(SPEC_ERR_ARG, "null uniforms");
    int rc = m->ensure_sampling();
    if (rc) return rc;
  }
  if (m->host_dirty) return fail(SPEC_ERR_STATE, "call spec_sync_seqs after device-resident steps");
  const int K = m->K, mb = m->cfg.max_batch;
  for (int s = 0; s < n_seq; ++s) {
    const int q = seq_ids[s];
    if (!m->seq_ok(q)) return fail(SPEC_ERR_ARG, "sequence " + std::to_string(q) + " not prefilled");
    for (int t = 0; t < s; ++t)
      if (seq_ids[t] == q) return fail(SPEC_ERR_ARG, "duplicate sequence in batch");
    const int nd = n_draft ? n_draft[s] : K;
    if (nd < 0 || nd > K) return fail(SPEC_ERR_ARG, "n_draft out of range");
    for (int j = 0; j < K; ++j) {
      const int d = drafts[s * K + j];
      if (j < nd && (d < 0 || d >= m->cfg.vocab)) return fail(SPEC_ERR_ARG, "draft token out of range");
    }
    if (m->seq_len_h[q] + m->R > m->cfg.max_ctx) return fail(SPEC_ERR_ARG, "sequence reached max_ctx");
  }
  // a0: pages for positions n .. n+K of every sequence
  for (int s = 0; s < n_seq; ++s) {
    const int q = seq_ids[s];
    const size_t before = m->pool->table(q).size();
    int rc = m->pool->reserve(q, m->seq_len_h[q] + m->R);
    if (rc) return fail(rc, "KV pool exhausted");
    if (m->pool->table(q).size() != before && (rc = m->push_table(q))) return rc;
  }
  std::fill(m->pin_in, m->pin_in + 4 + m->step_in_n, 0);    // out_ptrs = 0: results go to step_out
  int32_t* in = m->pin_in + 4;
  for (int s = 0; s < n_seq; ++s) {
    in[s] = seq_ids[s];
    const int nd = n_draft ? n_draft[s] : K;
    for (int j = 0; j < K; ++j) in[mb + s * K + j] = (j < nd && drafts) ? drafts[s * K + j] : 0;
    in[mb + mb * K + s] = nd;
  }
  CU(cudaMemcpyAsync(m->B.out_ptrs, m->pin_in, (4 + m->step_in_n) * sizeof(int32_t), cudaMemcpyHostToDevice,
                     m->stream));
  m->h2d_bytes += (int64_t)(4 + m->step_in_n) * sizeof(int32_t);
  if (smp) {
    const size_t ua_n = (size_t)mb * K, us_n = (size_t)mb * m->R, nin = ua_n + us_n + 1;
    std::fill(m->pin_smp, m->pin_smp + nin, 0.f);
    if (K > 0) std::copy(smp->u_accept, smp->u_accept + (size_t)n_seq * K, m->pin_smp);
    std::copy(smp->u_sample, smp->u_sample + (size_t)n_seq * m->R, m->pin_smp + ua_n);
    m->pin_smp[ua_n + us_n] = 1.f / smp->temperature;
    CU(cudaMemcpyAsync(m->smp_in, m->pin_smp, nin * sizeof(float), cudaMemcpyHostToDevice, m->stream));
    m->h2d_bytes += (int64_t)(nin * sizeof(float));
  }
  if (logits_dev) {
    mtp_forget_steps(m);
    m->enqueue_verify(n_seq, logits_dev, false);
    CU(cudaStreamSynchronize(m->stream));
    CU(cudaGetLastError());
    return m->check_err();
  }
  cudaGraphExec_t ge;
  int rc = m->graph_for(n_seq, &ge, smp != nullptr);
  if (rc) return rc;
  CU(cudaGraphLaunch(ge, m->stream));
  CU(cudaMemcpyAsync(m->pin_out, m->B.step_out, m->step_out_n * sizeof(int32_t), cudaMemcpyDeviceToHost,
                     m->stream));
  m->d2h_bytes += (int64_t)m->step_out_n * sizeof(int32_t);
  CU(cudaStreamSynchronize(m->stream));
  if (m->pin_out[2 * mb] != 0) {   // device error bits, copied by the commit kernel
    CU(cudaMemsetAsync(m->S.err, 0, sizeof(int), m->stream));
    CU(cudaStreamSynchronize(m->stream));
    return fail(SPEC_ERR_STATE, "device error bits " + std::to_string(m->pin_out[2 * mb]) +
                                    " (1 page, 2 token, 4 position out of range); step not committed on the host");
  }
  mtp_forget_steps(m);
  for (int s = 0; s < n_seq; ++s) {
    const int q = seq_ids[s];
    if (m->mtp) {   // the draft head reads this step's rows of q: row 0 at position seq_len_h[q]
      m->mtp->last_idx[q] = s;
      m->mtp->last_pos0[q] = m->seq_len_h[q];
    }
    const int a = m->pin_out[s], bonus = m->pin_out[mb + s];
    const int nd = n_draft ? n_draft[s] : K;
    for (int j = 0; j < a; ++j) m->gen[q].push_back(drafts[s * K + j]);
    m->gen[q].push_back(bonus);
    m->seq_len_h[q] += a + 1;
    m->last_tok_h[q] = bonus;
    // mirror the device-side trim of the block table
    m->pool->commit(q, m->seq_len_h[q], m->keep_h[q]);
    int32_t* row = m->bt_h.data() + (size_t)q * m->D.max_pages;
    const auto& t = m->pool->table(q);
    std::fill(row, row + m->D.max_pages, -1);
    std::copy(t.begin(), t.end(), row);
    (void)nd;
    if (out_acc) out_acc[s] = a;
    if (out_bonus) out_bonus[s] = bonus;
  }
  return SPEC_OK;
}

int spec_verify_step(spec_model* m, int32_t seq_id, const int32_t* draft_tokens, int n_draft,
                     int32_t* out_accepted_len, int32_t* out_bonus_token) {
  if (!m) return fail(SPEC_ERR_ARG, "null model");
  if (n_draft < 0 || n_draft > m->K || (n_draft > 0 && !draft_tokens)) return fail(SPEC_ERR_ARG, "bad drafts");
  std::vector<int32_t> d(std::max(m->K, 1), 0);
  for (int j = 0; j < n_draft; ++j) d[j] = draft_tokens[j];
  return verify_host(m, 1, &seq_id, d.data(), &n_draft, out_accepted_len, out_bonus_token, nullptr);
}

int spec_verify_step_batch(spec_model* m, int n_seq, const int32_t* seq_ids, const int32_t* drafts,
                           const int32_t* n_draft, int32_t* out_accepted, int32_t* out_bonus) {
  if (!out_accepted || !out_bonus) return fail(SPEC_ERR_ARG, "null outputs");
  return verify_host(m, n_seq, seq_ids, drafts, n_draft, out_accepted, out_bonus, nullptr);
}

int spec_verify_step_sample_batch(spec_model* m, int n_seq, const int32_t* seq_ids, const int32_t* drafts,
                                  const int32_t* n_draft, const float* u_accept, const float* u_sample,
                                  float temperature, int32_t* out_accepted, int32_t* out_token) {
  if (!out_accepted || !out_token) return fail(SPEC_ERR_ARG, "null outputs");
  const SampleArgs smp{u_accept, u_sample, temperature};
  return verify_host(m, n_seq, seq_ids, drafts, n_draft, out_accepted, out_token, nullptr, &smp);
}

int spec_verify_step_sample_dev(spec_model* m, int n_seq, const int32_t* seq_ids_dev, const int32_t* drafts_dev,
                                const int32_t* n_draft_dev, const float* u_accept_dev, const float* u_sample_dev,
                                float temperature, int32_t* out_accepted_dev, int32_t* out_token_dev) {
  if (!m || n_seq < 1 || n_seq > m->cfg.max_batch || !seq_ids_dev || !n_draft_dev ||
      (m->K > 0 && (!drafts_dev || !u_accept_dev)) || !u_sample_dev || !out_accepted_dev || !out_token_dev)
    return fail(SPEC_ERR_ARG, "bad device step arguments");
  if (!(temperature > 0.f) || !std::isfinite(1.f / temperature)) return fail(SPEC_ERR_ARG, "temperature must be positive");
  int rc = m->ensure_sampling();
  if (rc) return rc;
  cudaGraphExec_t ge;
  if ((rc = m->graph_for(n_seq, &ge, true))) return rc;
  launch_stage_dev(m->B, n_seq, m->K, seq_ids_dev, drafts_dev, n_draft_dev, out_accepted_dev, out_token_dev,
                   m->stream);
  launch_stage_sample(m->smp_in, m->cfg.max_batch, m->K, u_accept_dev, u_sample_dev, n_seq, 1.f / temperature,
                      m->stream);
  CU(cudaGraphLaunch(ge, m->stream));
  m->host_dirty = true;
  mtp_forget_steps(m);
  return SPEC_OK;
}

int spec_debug_logits(spec_model* m, int n_seq, const int32_t* seq_ids, const int32_t* drafts, float* logits_dev) {
  if (!logits_dev) return fail(SPEC_ERR_ARG, "null logits buffer");
  return verify_host(m, n_seq, seq_ids, drafts, nullptr, nullptr, nullptr, logits_dev);
}

int spec_verify_step_batch_dev(spec_model* m, int n_seq, const int32_t* seq_ids_dev, const int32_t* drafts_dev,
                               const int32_t* n_draft_dev, int32_t* out_accepted_dev, int32_t* out_bonus_dev) {
  if (!m || n_seq < 1 || n_seq > m->cfg.max_batch || !seq_ids_dev || !n_draft_dev ||
      (m->K > 0 && !drafts_dev) || !out_accepted_dev || !out_bonus_dev)
    return fail(SPEC_ERR_ARG, "bad device step arguments");
  cudaGraphExec_t ge;
  int rc = m->graph_for(n_seq, &ge);
  if (rc) return rc;
  launch_stage_dev(m->B, n_seq, m->K, seq_ids_dev, drafts_dev, n_draft_dev, out_accepted_dev, out_bonus_dev,
                   m->stream);
  CU(cudaGraphLaunch(ge, m->stream));
  m->host_dirty = true;
  mtp_forget_steps(m);
  return SPEC_OK;
}

// Host-side gate for the profiler: the stream waits in this host function
// until every launch of the step is enqueued, so the events around each kernel
// time the kernel rather than the host's enqueue latency. Bounded wait.
static void CUDART_CB profile_gate(void* arg) {
  auto* flag = static_cast<std::atomic<int>*>(arg);
  for (int i = 0; i < 20000 && flag->load() == 0; ++i) std::this_thread::sleep_for(std::chrono::microseconds(100));
}

int spec_profile_steps_dev(spec_model* m, int n_seq, const int32_t* seq_ids_dev, const int32_t* drafts_dev,
                           const int32_t* n_draft_dev, int n_steps, int drafts_step_stride, spec_kernel_stat* out,
                           int n_out) {
  if (!m || n_seq < 1 || n_seq > m->cfg.max_batch || n_steps < 1 || !out || n_out < 1 || !seq_ids_dev ||
      !n_draft_dev || (m->K > 0 && !drafts_dev))
    return fail(SPEC_ERR_ARG, "bad profile arguments");
  const int per_step = launches_per_step(m->D, n_seq * m->R) + 1;
  spec_model::Prof p;
  p.ev.resize(2 * per_step);
  p.cls.resize(per_step);
  for (auto& e : p.ev) CU(cudaEventCreate(&e));
  CU(cudaMallocHost(&p.act, m->D.L * sizeof(int32_t)));
  struct PdlOff {
    bool saved;
    PdlOff() : saved(pdl_enabled()) { pdl_enabled() = false; }   // events bracket single kernels
    ~PdlOff() { pdl_enabled() = saved; }
  } pdl_off;
  std::vector<double> ms(KC_COUNT, 0.0);
  std::vector<int64_t> launches(KC_COUNT, 0), units(KC_COUNT, 0);
  int rc = SPEC_OK;
  for (int s = 0; s < n_steps && rc == SPEC_OK; ++s) {
    p.n = 0;
    p.nact = 0;
    m->prof_gate.store(0);
    CU(cudaLaunchHostFunc(m->stream, profile_gate, &m->prof_gate));
    const int32_t* d = drafts_dev ? drafts_dev + (size_t)s * drafts_step_stride : nullptr;
    m->run_k(&p, KC_STAGE,
             [&] { launch_stage_dev(m->B, n_seq, m->K, seq_ids_dev, d, n_draft_dev, nullptr, nullptr, m->stream); });
    m->enqueue_verify(n_seq, nullptr, true, &p);
    m->prof_gate.store(1);
    cudaError_t e = cudaStreamSynchronize(m->stream);
    if (e != cudaSuccess) { rc = fail(SPEC_ERR_CUDA, cudaGetErrorString(e)); break; }
    for (int i = 0; i < p.n; ++i) {
      float t = 0.f;
      cudaEventElapsedTime(&t, p.ev[2 * i], p.ev[2 * i + 1]);
      ms[p.cls[i]] += t;
      launches[p.cls[i]] += 1;
    }
    for (int i = 0; i < p.nact; ++i) {
      units[KC_GATEUP] += p.act[i];
      units[KC_DOWN] += p.act[i];
    }
  }
  for (auto& e : p.ev) cudaEventDestroy(e);
  cudaFreeHost(p.act);
  m->host_dirty = true;
  if (rc) return rc;
  for (int i = 0; i < std::min(n_out, (int)KC_COUNT); ++i) {
    out[i].ms = (float)ms[i];
    out[i].launches = (int32_t)launches[i];
    out[i].units = units[i];
  }
  return std::min(n_out, (int)KC_COUNT);
}

const char* spec_kernel_class_name(int cls) {
  static const char* names[KC_COUNT] = {"assemble", "qkv_rope_kvwrite", "attn_splitkv_merge", "oproj_residual",
                                        "router_topk_permute", "expert_gateup_swiglu", "expert_down",
                                        "expert_combine", "lmhead_argmax_commit", "accept_commit", "stage_inputs"};
  return (cls >= 0 && cls < KC_COUNT) ? names[cls] : "";
}

int spec_io_bytes(spec_model* m, int64_t* out_h2d, int64_t* out_d2h) {
  if (!m) return fail(SPEC_ERR_ARG, "null model");
  if (out_h2d) *out_h2d = m->h2d_bytes;
  if (out_d2h) *out_d2h = m->d2h_bytes;
  return SPEC_OK;
}

int spec_reserve_seq(spec_model* m, int32_t seq_id, int n_tokens) {
  if (!m || !m->seq_ok(seq_id) || n_tokens < 0 || n_tokens > m->cfg.max_ctx) return fail(SPEC_ERR_ARG, "bad reserve");
  if (m->host_dirty) return fail(SPEC_ERR_STATE, "call spec_sync_seqs after device-resident steps");
  int rc = m->pool->reserve(seq_id, n_tokens);
  if (rc) return fail(rc, "KV pool exhausted");
  m->keep_h[seq_id] = KvPool::pages_for(n_tokens, m->cfg.page_size);
  if ((rc = m->push_table(seq_id)) || (rc = m->push_seq_scalars(seq_id))) return rc;
  CU(cudaStreamSynchronize(m->stream));
  return SPEC_OK;
}

int spec_sync_seqs(spec_model* m) {
  if (!m) return fail(SPEC_ERR_ARG, "null model");
  CU(cudaStreamSynchronize(m->stream));
  int rc = m->check_err();
  if (rc) return rc;
  const int ns = m->cfg.max_seqs;
  std::vector<int32_t> len(ns), last(ns), nout(ns);
  CU(cudaMemcpy(len.data(), m->S.seq_len, ns * 4, cudaMemcpyDeviceToHost));
  CU(cudaMemcpy(last.data(), m->S.last_tok, ns * 4, cudaMemcpyDeviceToHost));
  CU(cudaMemcpy(nout.data(), m->S.n_out, ns * 4, cudaMemcpyDeviceToHost));
  for (int q = 0; q < ns; ++q) {
    if (!m->busy[q]) continue;
    const int n = std::min(nout[q], m->cfg.max_ctx);
    m->gen[q].resize(n);
    if (n) CU(cudaMemcpy(m->gen[q].data(), m->S.out_tok + (size_t)q * m->cfg.max_ctx, n * 4, cudaMemcpyDeviceToHost));
    m->seq_len_h[q] = len[q];
    m->last_tok_h[q] = last[q];
    m->pool->commit(q, len[q], m->keep_h[q]);
    int32_t* row = m->bt_h.data() + (size_t)q * m->D.max_pages;
    const auto& t = m->pool->table(q);
    std::fill(row, row + m->D.max_pages, -1);
    std::copy(t.begin(), t.end(), row);
  }
  m->host_dirty = false;
  return SPEC_OK;
}

int spec_release_seq(spec_model* m, int32_t seq_id) {
  if (!m || !m->seq_ok(seq_id)) return fail(SPEC_ERR_ARG, "sequence not active");
  if (m->host_dirty) return fail(SPEC_ERR_STATE, "call spec_sync_seqs after device-resident steps");
  m->pool->release(seq_id);
  if (m->mtp) {   // the draft head's caches of this sequence
    MtpHead& H = *m->mtp;
    for (int k = 0; k < H.Kmax; ++k) H.blk->pool->release(seq_id * H.Kmax + k);
    H.p0[seq_id] = -1;
    H.last_idx[seq_id] = -1;
  }
  m->busy[seq_id] = 0;
  m->seq_len_h[seq_id] = 0;
  m->keep_h[seq_id] = 0;
  m->gen[seq_id].clear();
  int rc = m->push_table(seq_id);
  if (rc) return rc;
  if ((rc = m->push_seq_scalars(seq_id))) return rc;
  CU(cudaStreamSynchronize(m->stream));
  return SPEC_OK;
}

int spec_seq_info(spec_model* m, int32_t seq_id, int32_t* out_len, int32_t* out_n_generated) {
  if (!m || !m->seq_ok(seq_id)) return fail(SPEC_ERR_ARG, "sequence not active");
  if (out_len) *out_len = m->seq_len_h[seq_id];
  if (out_n_generated) *out_n_generated = (int32_t)m->gen[seq_id].size();
  return SPEC_OK;
}

int spec_seq_tokens(spec_model* m, int32_t seq_id, int32_t* out_tokens, int cap) {
  if (!m || !m->seq_ok(seq_id) || !out_tokens || cap < 0) return fail(SPEC_ERR_ARG, "bad arguments");
  const auto& g = m->gen[seq_id];
  const int n = std::min<int>(cap, (int)g.size());
  std::copy(g.begin(), g.begin() + n, out_tokens);
  return n;
}

int spec_seq_block_table(spec_model* m, int32_t seq_id, int32_t* out_pages, int cap, int32_t* out_n) {
  if (!m || seq_id < 0 || seq_id >= m->n_slots || !out_pages || cap < 0) return fail(SPEC_ERR_ARG, "bad arguments");
  std::vector<int32_t> row(m->D.max_pages);
  CU(cudaStreamSynchronize(m->stream));
  CU(cudaMemcpy(row.data(), m->S.bt + (size_t)seq_id * m->D.max_pages, m->D.max_pages * 4, cudaMemcpyDeviceToHost));
  int n = 0;
  while (n < m->D.max_pages && row[n] >= 0) ++n;
  for (int i = 0; i < std::min(cap, m->D.max_pages); ++i) out_pages[i] = row[i];
  if (out_n) *out_n = n;
  return SPEC_OK;
}

int spec_free_pages(spec_model* m) {
  if (!m) return fail(SPEC_ERR_ARG, "null model");
  return m->pool->free_count();
}

int spec_step_launches(spec_model* m, int n_seq) {
  if (!m || n_seq < 1) return fail(SPEC_ERR_ARG, "bad arguments");
  const int merge = attn_separate_merge(m->D, m->R, n_seq * m->R) ? m->D.L : 0;   // + the standalone attention merges
  if (m->use_tc)   // per layer: norm, QKV, RoPE/KV, attention, O, router, gather, gate/up, down, combine
    return 1 + m->D.L * 10 + 3 + merge;
  return launches_per_step(m->D, n_seq * m->R) + merge;
}

// ---- FastMTP draft head -----------------------------------------------------
int spec_mtp_init(spec_model* m, const void* const* host_tensors, int inter) {
  if (!m || !host_tensors || inter < 4) return fail(SPEC_ERR_ARG, "bad draft-head arguments");
  if (m->mtp) return fail(SPEC_ERR_STATE, "the model already has a draft head");
  if (m->K < 1) return fail(SPEC_ERR_ARG, "a draft head needs max_draft >= 1");
  for (int i = 0; i < 13; ++i)
    if (!host_tensors[i]) return fail(SPEC_ERR_ARG, "missing draft-head tensor " + std::to_string(i));
  const spec_config& c = m->cfg;
  std::unique_ptr<MtpHead> H(new MtpHead());
  H->Kmax = m->K;
  H->R = 2 * m->K;                      // a depth's rows per call: a + k <= 2 K
  H->B0 = 256;
  H->ymax = H->B0 + 2 * m->K;
  H->pass_ints = 4 * H->R + H->R * (int)(sizeof(float*) / sizeof(int));
  H->max_pass = H->Kmax * ((H->ymax + H->R - 1) / H->R);
  spec_config bc = c;                   // the draft block: one layer, dense SwiGLU of width `inter`
  bc.n_layers = 1;
  bc.n_experts = 0;
  bc.top_k = 0;
  bc.n_shared = 1;
  bc.inter = inter;
  bc.wdtype = c.wdtype == SPEC_F32 ? SPEC_F32 : SPEC_BF16;
  bc.max_seqs = c.max_seqs * m->K;
  bc.max_batch = 1;
  bc.max_draft = H->R - 1;
  bc.max_ctx = c.max_ctx + 2 * H->R;
  bc.n_pages = bc.max_seqs * ((bc.max_ctx + c.page_size - 1) / c.page_size + 1) + 8;
  bc.prefill_chunk = H->R;
  // tensor list of the block model: tok_embed, final_norm, lm_head (tied), then one layer
  const void* null = nullptr;
  const void* bt[N_GLOBAL + PER_LAYER] = {host_tensors[0], host_tensors[1], host_tensors[2],
                                          host_tensors[6], host_tensors[7], null, host_tensors[8], null,
                                          host_tensors[9], null, host_tensors[10], null, host_tensors[11], null,
                                          host_tensors[12], null};
  spec_model* blk = nullptr;
  int rc = spec_init_model(&bc, bt, reinterpret_cast<uintptr_t>(m->stream), &blk);
  if (rc) return rc;
  H->blk = blk;
  if (blk->use_tc) return fail(SPEC_ERR_UNSUPPORTED, "draft head: more than 4 drafts per step");
  const int h = c.hidden, welt = c.wdtype == SPEC_F32 ? 4 : 2;
  auto dal = [&](void** q, size_t bytes) -> int {
    if (cudaMalloc(q, bytes ? bytes : 1) != cudaSuccess) return fail(SPEC_ERR_NOMEM, "draft head allocation");
    H->allocs.push_back(*q);
    return SPEC_OK;
  };
  if ((rc = dal((void**)&H->enorm, h * 4)) || (rc = dal((void**)&H->hnorm, h * 4)) ||
      (rc = dal(&H->P, (size_t)h * 2 * h * welt)) || (rc = dal((void**)&H->cat, (size_t)H->R * 2 * h * 4)) ||
      (rc = dal((void**)&H->Y, (size_t)H->Kmax * H->ymax * h * 4)) ||
      (rc = dal((void**)&H->ylast, (size_t)c.max_seqs * H->Kmax * h * 4)) ||
      (rc = dal((void**)&H->b0, (size_t)c.max_seqs * H->B0 * h * 4)) ||
      (rc = dal((void**)&H->d_meta, (size_t)H->pass_ints * 4)) || (rc = dal((void**)&H->d_drafts, H->Kmax * 4)))
    return rc;
  CU(cudaMemcpy(H->enorm, host_tensors[3], h * 4, cudaMemcpyHostToDevice));
  CU(cudaMemcpy(H->hnorm, host_tensors[4], h * 4, cudaMemcpyHostToDevice));
  CU(cudaMemcpy(H->P, host_tensors[5], (size_t)h * 2 * h * welt, cudaMemcpyHostToDevice));
  CU(cudaMallocHost(&H->pin, (size_t)H->max_pass * H->pass_ints * sizeof(int)));
  blk->B.row_rope = H->d_meta + 2 * H->R;
  H->p0.assign(c.max_seqs, -1);
  H->p_done.assign(c.max_seqs, -2);
  H->b0_rows.assign(c.max_seqs, 0);
  H->last_pos0.assign(c.max_seqs, -1);
  H->last_idx.assign(c.max_seqs, -1);
  H->prompt_tok.assign(c.max_seqs, {});
  m->mtp = H.release();
  return SPEC_OK;
}

static int mtp_draft(spec_model* m, int32_t seq_id, int K, int32_t* out_drafts, float* logits_dev,
                     float* states_dev = nullptr, int states_cap = 0, int32_t* out_n_states = nullptr) {
  if (!m || !out_drafts) return fail(SPEC_ERR_ARG, "null argument");
  if (!m->mtp) return fail(SPEC_ERR_STATE, "no draft head (spec_mtp_init)");
  if (!m->seq_ok(seq_id)) return fail(SPEC_ERR_ARG, "sequence not active");
  if (m->host_dirty) return fail(SPEC_ERR_STATE, "call spec_sync_seqs after device-resident steps");
  MtpHead& H = *m->mtp;
  if (K < 1 || K > H.Kmax) return fail(SPEC_ERR_ARG, "K out of range");
  const int p0 = H.p0[seq_id];
  if (p0 < 0) return fail(SPEC_ERR_UNSUPPORTED, "the draft head does not take sequences with a shared prefix");
  const int N = m->seq_len_h[seq_id], p = N - 1, done = H.p_done[seq_id];
  if (p <= done) return fail(SPEC_ERR_STATE, "no new committed rows since the last draft");
  // decoder state of committed row r (depth 1): the prompt rows kept at
  // prefill (first call), else the rows of the verify step just run
  const bool first = done < p0;
  if (first && p - p0 + 1 > H.b0_rows[seq_id])
    return fail(SPEC_ERR_STATE, "the first draft must follow the prefill (and the prompt tail fit the head)");
  if (!first && (H.last_idx[seq_id] < 0 || H.last_pos0[seq_id] != done + 1))
    return fail(SPEC_ERR_STATE, "draft right after the verify step that committed the new rows");
  spec_model* blk = H.blk;
  const int h = m->D.h, R = H.R;
  const std::vector<int32_t>& pt = H.prompt_tok[seq_id];
  const std::vector<int32_t>& gen = m->gen[seq_id];
  const int plen = (int)pt.size();
  // x_i: committed tokens, then the drafts as -(j + 1) (read on the device)
  auto tok_at = [&](int i) -> int32_t {
    if (i < plen) return pt[i];
    if (i - plen < (int)gen.size()) return gen[i - plen];
    return -(i - N);
  };
  auto dec_row = [&](int r) -> const float* {
    if (first) return H.b0 + ((size_t)seq_id * H.B0 + (r - p0)) * h;
    return m->B.x + ((size_t)H.last_idx[seq_id] * m->R + (r - (done + 1))) * h;
  };
  // Every depth advances over the new committed rows, so a shorter K leaves
  // no depth's cache behind; depths 1..K add their speculative rows up to
  // p + k - 1, whose last one gives d_k.
  if (states_dev) {   // debug: the decoder rows depth 1 reads in this call (rows max(done + 1, p0) .. p)
    const int r0 = std::max(done + 1, p0), n = p - r0 + 1;
    if (n > states_cap) return fail(SPEC_ERR_ARG, "states_dev holds fewer rows than the call reads");
    for (int r = r0; r <= p; ++r)
      CU(cudaMemcpyAsync(states_dev + (size_t)(r - r0) * h, dec_row(r), h * 4, cudaMemcpyDeviceToDevice, m->stream));
    *out_n_states = n;
  }
  std::vector<int> start(H.Kmax + 1, 0), last(H.Kmax + 1, -1);
  int npass = 0;
  for (int k = 1; k <= H.Kmax; ++k) {
    const int first_row = p0 + k - 1;            // cache index 0 of depth k
    const int s0 = std::max(done + 1, first_row), s1 = k <= K ? p + k - 1 : p;
    start[k] = s0;
    last[k] = s1;
    if (s1 < s0) continue;
    if (s1 - s0 + 1 > H.ymax) return fail(SPEC_ERR_UNSUPPORTED, "draft head: too many new rows");
    const int slot = seq_id * H.Kmax + (k - 1);
    int rc = blk->pool->reserve(slot, s0 + ((s1 - s0) / R + 1) * R - first_row);
    if (rc) return fail(rc, "draft head: KV pool exhausted");
    if ((rc = blk->push_table(slot))) return rc;
    float* Yk = H.Y + (size_t)(k - 1) * H.ymax * h;
    for (int ps = s0; ps <= s1; ps += R, ++npass) {
      if (npass >= H.max_pass) return fail(SPEC_ERR_UNSUPPORTED, "draft head: too many passes");
      const int nreal = std::min(R, s1 - ps + 1);
      int* meta = H.pin + (size_t)npass * H.pass_ints;
      const float** srcp = reinterpret_cast<const float**>(meta + 4 * R);
      for (int i = 0; i < R; ++i) {
        const int r = ps + i;
        const bool real = i < nreal;
        meta[i] = real ? tok_at(r + 1) : 0;                    // x_(r+1)
        meta[R + i] = r - first_row;                           // cache index
        meta[2 * R + i] = r;                                   // RoPE position
        meta[3 * R + i] = slot;
        const float* src = nullptr;
        if (real) {
          if (k == 1) src = dec_row(r);
          else if (r - 1 < start[k - 1]) src = H.ylast + ((size_t)seq_id * H.Kmax + (k - 2)) * h;   // kept row
          else src = H.Y + ((size_t)(k - 2) * H.ymax + (r - 1 - start[k - 1])) * h;
        }
        srcp[i] = src;
      }
      // the pinned area of each pass stays untouched until the call's final sync
      CU(cudaMemcpyAsync(H.d_meta, meta, H.pass_ints * sizeof(int), cudaMemcpyHostToDevice, m->stream));
      CU(cudaMemcpyAsync(blk->B.row_pos, H.d_meta + R, R * 4, cudaMemcpyDeviceToDevice, m->stream));
      CU(cudaMemcpyAsync(blk->B.row_seq, H.d_meta + 3 * R, R * 4, cudaMemcpyDeviceToDevice, m->stream));
      launch_mtp_input(blk->D, H.d_meta, reinterpret_cast<const float* const*>(H.d_meta + 4 * R), H.d_drafts, R,
                       blk->tok_embed, H.enorm, blk->final_norm, H.hnorm, H.P, H.cat, blk->B.x, m->stream);
      const float* y = blk->enqueue_layers(R, R);
      CU(cudaMemcpyAsync(Yk + (size_t)(ps - s0) * h, y, (size_t)nreal * h * 4, cudaMemcpyDeviceToDevice, m->stream));
    }
    if (k <= K) {
      // d_k: greedy token of N_o(y) at row p + k - 1, the depth's last row
      blk->enqueue_lmhead(Yk + (size_t)(s1 - s0) * h, 1, logits_dev ? logits_dev + (size_t)(k - 1) * m->D.V : nullptr,
                          false, 0);
      CU(cudaMemcpyAsync(H.d_drafts + (k - 1), blk->B.g, 4, cudaMemcpyDeviceToDevice, m->stream));
    }
  }
  // keep each depth's row p for the next call
  for (int k = 1; k <= H.Kmax; ++k)
    if (p >= start[k] && p <= last[k])
      CU(cudaMemcpyAsync(H.ylast + ((size_t)seq_id * H.Kmax + (k - 1)) * h,
                         H.Y + ((size_t)(k - 1) * H.ymax + (p - start[k])) * h, h * 4, cudaMemcpyDeviceToDevice,
                         m->stream));
  int32_t* dout = blk->pin_out;
  CU(cudaMemcpyAsync(dout, H.d_drafts, K * 4, cudaMemcpyDeviceToHost, m->stream));
  CU(cudaStreamSynchronize(m->stream));
  CU(cudaGetLastError());
  int rc = blk->check_err();
  if (rc) return rc;
  H.p_done[seq_id] = p;
  for (int k = 0; k < K; ++k) out_drafts[k] = dout[k];
  return SPEC_OK;
}

int spec_mtp_draft(spec_model* m, int32_t seq_id, int K, int32_t* out_drafts) {
  return mtp_draft(m, seq_id, K, out_drafts, nullptr);
}

int spec_mtp_debug_draft(spec_model* m, int32_t seq_id, int K, int32_t* out_drafts, float* logits_dev,
                         float* states_dev, int states_cap, int32_t* out_n_states) {
  if (!logits_dev || !states_dev || !out_n_states) return fail(SPEC_ERR_ARG, "null debug output");
  return mtp_draft(m, seq_id, K, out_drafts, logits_dev, states_dev, states_cap, out_n_states);
}

// ---- host-only allocator entry points --------------------------------------
struct spec_pool { KvPool p; spec_pool(int a, int b, int c, int d) : p(a, b, c, d) {} };

int spec_pool_create(int n_pages, int page_size, int max_seqs, int max_pages_per_seq, spec_pool** out) {
  if (!out || n_pages < 1 || page_size < 1 || max_seqs < 1 || max_pages_per_seq < 1)
    return fail(SPEC_ERR_ARG, "bad pool shape");
  *out = new spec_pool(n_pages, page_size, max_seqs, max_pages_per_seq);
  return SPEC_OK;
}
int spec_pool_destroy(spec_pool* p) { delete p; return SPEC_OK; }
int spec_pool_reserve(spec_pool* p, int32_t seq, int n_tokens) {
  return p ? p->p.reserve(seq, n_tokens) : SPEC_ERR_ARG;
}
int spec_pool_commit(spec_pool* p, int32_t seq, int new_len, int keep_pages) {
  return p ? p->p.commit(seq, new_len, keep_pages) : SPEC_ERR_ARG;
}
int spec_pool_release(spec_pool* p, int32_t seq) { return p ? p->p.release(seq) : SPEC_ERR_ARG; }
int spec_pool_share(spec_pool* p, int32_t src_seq, int n_pages, int32_t dst) {
  return p ? p->p.share(src_seq, n_pages, dst) : SPEC_ERR_ARG;
}
int spec_pool_block_table(spec_pool* p, int32_t seq, int32_t* out, int cap, int32_t* out_n) {
  if (!p || !p->p.valid_seq(seq) || !out) return SPEC_ERR_ARG;
  const auto& t = p->p.table(seq);
  const int n = std::min<int>(cap, (int)t.size());
  std::copy(t.begin(), t.begin() + n, out);
  if (out_n) *out_n = (int32_t)t.size();
  return SPEC_OK;
}
int spec_pool_refcount(spec_pool* p, int32_t page) { return p ? p->p.refcount(page) : SPEC_ERR_ARG; }
int spec_pool_free_count(spec_pool* p) { return p ? p->p.free_count() : SPEC_ERR_ARG; }

}  // extern "C"
