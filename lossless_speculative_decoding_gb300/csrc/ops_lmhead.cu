// Kernel-level entry point: final RMSNorm + LM head + greedy argmax over the
// vocabulary for T activation rows, without materialising the logits.
#include <cuda_runtime.h>

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
  Dims D;
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

