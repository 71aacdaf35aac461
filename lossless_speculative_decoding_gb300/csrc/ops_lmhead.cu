// Kernel-level entry point: final RMSNorm + LM head + greedy argmax over the
// vocabulary for T activation rows, without materialising the logits.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/spec.h"
#include "kernels.h"

using namespace spec;

namespace {

int op_fail(int code, const char* msg) { return set_last_error(code, msg); }

// Shapes for the LM-head kernels: only h, V, eps and the weight type matter.
void lmhead_setup(int T, int h, int V, int w_dtype, float eps, Dims* D, StepBuf* B) {
  *D = Dims{};
  D->h = h;
  D->V = V;
  D->eps = eps;
  D->act_f32 = w_dtype == SPEC_F32;
  *B = StepBuf{};
  B->n_vblocks = (V + GEMV_WARPS * 4 - 1) / (GEMV_WARPS * 4);
  (void)T;
}

int check_lmhead_args(const float* x, int T, int h, int V, const void* w, int w_dtype, const float* gamma,
                      int32_t* out) {
  if (!x || !w || !gamma || !out) return op_fail(SPEC_ERR_ARG, "null pointer argument");
  if (T < 1 || h < 64 || V < 4) return op_fail(SPEC_ERR_ARG, "T >= 1, hidden >= 64 and vocab >= 4 required");
  if (w_dtype != SPEC_F32 && w_dtype != SPEC_BF16) return op_fail(SPEC_ERR_ARG, "LM head dtype must be F32 or BF16");
  if (V % 4 || (h * (w_dtype == SPEC_F32 ? 4 : 2)) % 16 || h % 4)
    return op_fail(SPEC_ERR_UNSUPPORTED, "vocab must be a multiple of 4 and a row a multiple of 16 bytes");
  if (h > 12288) return op_fail(SPEC_ERR_UNSUPPORTED, "hidden above 12288");
  return SPEC_OK;
}

}  // namespace

extern "C" {

int64_t spec_lmhead_argmax_scratch_bytes(int T, int V) {
  if (T < 1 || V < 4) return SPEC_ERR_ARG;
  const int64_t nvb = (V + GEMV_WARPS * 4 - 1) / (GEMV_WARPS * 4);
  return (int64_t)T * nvb * 8;
}

int spec_lmhead_argmax(const float* x_dev, int T, int hidden, int vocab, const void* w_dev, int w_dtype,
                       const float* gamma_dev, float eps, void* scratch_dev, size_t scratch_bytes,
                       int32_t* out_tokens_dev, uintptr_t cuda_stream) {
  int rc = check_lmhead_args(x_dev, T, hidden, vocab, w_dev, w_dtype, gamma_dev, out_tokens_dev);
  if (rc) return rc;
  if (!scratch_dev || (int64_t)scratch_bytes < spec_lmhead_argmax_scratch_bytes(T, vocab))
    return op_fail(SPEC_ERR_ARG, "scratch smaller than spec_lmhead_argmax_scratch_bytes(T, vocab)");
  if (configure_gemv_kernels() != cudaSuccess) return op_fail(SPEC_ERR_CUDA, "kernel attribute set-up failed");
  Dims D{};
  StepBuf B;
  lmhead_setup(T, hidden, vocab, w_dtype, eps, &D, &B);
  B.am_val = reinterpret_cast<float*>(scratch_dev);
  B.am_idx = reinterpret_cast<int*>(B.am_val + (size_t)T * B.n_vblocks);
  B.g = out_tokens_dev;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(cuda_stream);
  launch_lmhead(D, B, w_dev, gamma_dev, x_dev, T, nullptr, false, st);
  launch_argmax(B, T, st);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return op_fail(SPEC_ERR_CUDA, cudaGetErrorString(e));
  return SPEC_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free variant. Some callers cannot allocate device memory while
// they run: code inside a memory-pool-free real-time loop, or a host that
// owns every allocation itself and forbids libraries from calling
// cudaMalloc. For them the candidate scratch lives in this file-scope device
// array: every GPU that loads the library holds it until the process exits,
// and all calls on a device share it.
namespace {

constexpr int64_t kNoAllocPairs = SPEC_LMHEAD_NOALLOC_MAX_PAIRS;   // (max, index) candidates
static __device__ __align__(256) unsigned char g_lmhead_scratch[kNoAllocPairs * 8];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Once per device, with that device current: resolve the array's device
// address (host code cannot use the symbol itself) and set kernel attributes.
int noalloc_setup(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return op_fail(SPEC_ERR_CUDA, cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return op_fail(SPEC_ERR_UNSUPPORTED, "device index above 63");
  std::lock_guard<std::mutex> lk(g_setup_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_lmhead_scratch);
    if (e != cudaSuccess) return op_fail(SPEC_ERR_CUDA, cudaGetErrorString(e));
    if (configure_gemv_kernels() != cudaSuccess) return op_fail(SPEC_ERR_CUDA, "kernel attribute set-up failed");
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return SPEC_OK;
}

}  // namespace

extern "C" int spec_lmhead_argmax_noalloc(const float* x_dev, int T, int hidden, int vocab, const void* w_dev,
                                          int w_dtype, const float* gamma_dev, float eps,
                                          int32_t* out_tokens_dev, uintptr_t cuda_stream) {
  int rc = check_lmhead_args(x_dev, T, hidden, vocab, w_dev, w_dtype, gamma_dev, out_tokens_dev);
  if (rc) return rc;
  if (spec_lmhead_argmax_scratch_bytes(T, vocab) > kNoAllocPairs * 8)
    return op_fail(SPEC_ERR_ARG, "T * ceil(vocab / 32) exceeds SPEC_LMHEAD_NOALLOC_MAX_PAIRS");
  void* scratch = nullptr;
  if ((rc = noalloc_setup(&scratch))) return rc;
  Dims D{};
  StepBuf B;
  lmhead_setup(T, hidden, vocab, w_dtype, eps, &D, &B);
  // every candidate slot is written by its block before the reduction reads
  // it, so nothing has to be cleared between calls
  B.am_val = reinterpret_cast<float*>(scratch);
  B.am_idx = reinterpret_cast<int*>(B.am_val + (size_t)T * B.n_vblocks);
  B.g = out_tokens_dev;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(cuda_stream);
  launch_lmhead(D, B, w_dev, gamma_dev, x_dev, T, nullptr, false, st);
  launch_argmax(B, T, st);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return op_fail(SPEC_ERR_CUDA, cudaGetErrorString(e));
  return SPEC_OK;
}
