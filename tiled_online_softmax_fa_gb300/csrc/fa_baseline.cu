// fa_baseline.cu -- the materialised attention baseline, in a library of its own
// (libfa_baseline.so) so that the tiled forward library links no BLAS.
//
// The baseline is the pages' `standard_attention` (aiml.sh "Speed up long contexts with
// FlashAttention", lab.py) on the GPU: the N x N scores and probabilities live in device
// memory.  S = scale Q K^T and acc = P V are plain cuBLAS batched GEMMs; the row softmax
// and the normalisation are this library's kernels (fa_materialised_kernel.cuh).  It is
// the contrast arm that the tiled kernels are measured against, not a fast path.
#include <cublas_v2.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstdio>
#include <mutex>
#include <string>

#include "../../include/fa_baseline.h"
#include "fa_materialised_kernel.cuh"

namespace {

constexpr int kMaxDevices = 64;

thread_local std::string t_last_error;
std::mutex g_mu;

int set_error(int status, const std::string& msg) {
  t_last_error = msg;
  return status;
}

int cuda_error(const char* what, cudaError_t e) {
  return set_error(FA_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

bool head_dim_ok(int64_t d) { return d == 16 || d == 32 || d == 64 || d == 128 || d == 256; }

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

// The current device, which must be compute capability 10.3.
int check_device(int* dev_index) {
  int dev = 0, major = 0, minor = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_error("cudaGetDevice", e);
  if (dev < 0 || dev >= kMaxDevices) return set_error(FA_ERR_UNSUPPORTED, "device index too large");
  if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
      (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
    return cuda_error("cudaDeviceGetAttribute", e);
  if (major != 10 || minor != 3) return set_error(FA_ERR_ARCH, "device is not sm_103 (GB300-class)");
  *dev_index = dev;
  return FA_OK;
}

cublasHandle_t g_cublas[kMaxDevices];

// Workspace layout: S fp32 [BH, N, N] | P bf16 [BH, N, N] | acc fp32 [BH, N, d] |
// l_round fp32 [BH, N] (each part starts on a 256-byte boundary).
int64_t round256(int64_t x) { return (x + 255) / 256 * 256; }
int64_t materialised_bytes(int64_t BH, int64_t N, int64_t d) {
  return round256(BH * N * N * 4) + round256(BH * N * N * 2) + round256(BH * N * d * 4) +
         round256(BH * N * 4);
}

int cublas_error(const char* what, cublasStatus_t st) {
  char buf[96];
  snprintf(buf, sizeof buf, "%s failed (cublasStatus %d)", what, static_cast<int>(st));
  return set_error(FA_ERR_CUDA, buf);
}

}  // namespace

extern "C" {

int64_t fa_materialised_workspace_bytes(int64_t B, int64_t H, int64_t N, int64_t d) {
  if (B < 0 || H < 0 || N < 0 || !head_dim_ok(d)) return -1;
  if (B == 0 || H == 0 || N == 0) return 0;
  if (B > INT32_MAX / H || N > (int64_t{1} << 20)) return -1;
  const int64_t BH = B * H;
  if (BH > (INT64_MAX / 8) / (N * N)) return -1;
  return materialised_bytes(BH, N, d);
}

int fa_fwd_materialised(const void* q, const void* k, const void* v, void* o, float* lse,
                        int64_t B, int64_t H, int64_t N, int64_t d, int causal, float scale,
                        void* workspace, size_t workspace_bytes_given, void* stream) {
  t_last_error.clear();
  if (B < 0 || H < 0 || N < 0) return set_error(FA_ERR_INVALID_ARG, "negative size");
  if (!head_dim_ok(d)) return set_error(FA_ERR_UNSUPPORTED, "head dim must be 16, 32, 64, 128 or 256");
  if (B == 0 || H == 0 || N == 0) return FA_OK;
  if (!q || !k || !v || !o) return set_error(FA_ERR_INVALID_ARG, "null tensor pointer");
  if (!std::isfinite(scale) || scale < 0.f)
    return set_error(FA_ERR_INVALID_ARG, "scale must be finite and >= 0");
  const int64_t need = fa_materialised_workspace_bytes(B, H, N, d);
  if (need < 0) return set_error(FA_ERR_UNSUPPORTED, "sizes beyond the materialised path's range");
  const int64_t BH = B * H;
  if (BH * N > INT32_MAX) return set_error(FA_ERR_UNSUPPORTED, "too many rows for the softmax grid");
  if (!workspace) return set_error(FA_ERR_INVALID_ARG, "the materialised path needs a workspace");
  if (static_cast<int64_t>(workspace_bytes_given) < need)
    return set_error(FA_ERR_INVALID_ARG, "workspace too small (see fa_materialised_workspace_bytes)");
  for (const void* ptr : {q, k, v, static_cast<const void*>(o)})
    if (reinterpret_cast<uintptr_t>(ptr) % 16 != 0)
      return set_error(FA_ERR_MISALIGNED, "tensor base address not 16-byte aligned");
  if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0)
    return set_error(FA_ERR_MISALIGNED, "workspace not 256-byte aligned");
  if (lse && reinterpret_cast<uintptr_t>(lse) % 4 != 0)
    return set_error(FA_ERR_MISALIGNED, "lse not 4-byte aligned");
  const size_t bytes = static_cast<size_t>(BH * N * d) * 2;
  const size_t lse_bytes = static_cast<size_t>(BH * N) * 4;
  for (const void* in : {q, k, v}) {
    if (overlaps(o, bytes, in, bytes)) return set_error(FA_ERR_INVALID_ARG, "o overlaps an input");
    if (lse && overlaps(lse, lse_bytes, in, bytes))
      return set_error(FA_ERR_INVALID_ARG, "lse overlaps an input");
  }
  if (lse && overlaps(lse, lse_bytes, o, bytes)) return set_error(FA_ERR_INVALID_ARG, "lse overlaps o");
  for (const void* t : {q, k, v, static_cast<const void*>(o)})
    if (overlaps(workspace, static_cast<size_t>(need), t, bytes))
      return set_error(FA_ERR_INVALID_ARG, "workspace overlaps a tensor");
  if (lse && overlaps(workspace, static_cast<size_t>(need), lse, lse_bytes))
    return set_error(FA_ERR_INVALID_ARG, "workspace overlaps lse");

  int dev_index = 0;
  const int st = check_device(&dev_index);
  if (st != FA_OK) return st;
  cudaError_t e;

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  float* S = reinterpret_cast<float*>(ws);
  __nv_bfloat16* P = reinterpret_cast<__nv_bfloat16*>(ws + round256(BH * N * N * 4));
  float* acc = reinterpret_cast<float*>(ws + round256(BH * N * N * 4) + round256(BH * N * N * 2));
  float* l_round = reinterpret_cast<float*>(ws + round256(BH * N * N * 4) + round256(BH * N * N * 2) +
                                            round256(BH * N * d * 4));
  const int n = static_cast<int>(N), dd = static_cast<int>(d);
  const long long sN2 = static_cast<long long>(N) * N, sNd = static_cast<long long>(N) * d;
  const float one = 1.f, zero = 0.f;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // one handle per device; the lock also serialises its stream binding across host threads
  std::lock_guard<std::mutex> lock(g_mu);
  cublasHandle_t& h = g_cublas[dev_index];
  cublasStatus_t cs;
  if (!h && (cs = cublasCreate(&h)) != CUBLAS_STATUS_SUCCESS) {
    h = nullptr;
    return cublas_error("cublasCreate", cs);
  }
  if ((cs = cublasSetStream(h, s)) != CUBLAS_STATUS_SUCCESS) return cublas_error("cublasSetStream", cs);
  // column-major view: S^T (N x N) = K (d x N)^T * Q (d x N), i.e. S[i][j] = scale q_i . k_j
  cs = cublasGemmStridedBatchedEx(h, CUBLAS_OP_T, CUBLAS_OP_N, n, n, dd, &scale, k, CUDA_R_16BF, dd,
                                  sNd, q, CUDA_R_16BF, dd, sNd, &zero, S, CUDA_R_32F, n, sN2,
                                  static_cast<int>(BH), CUBLAS_COMPUTE_32F, CUBLAS_GEMM_DEFAULT);
  if (cs != CUBLAS_STATUS_SUCCESS) return cublas_error("cublasGemmStridedBatchedEx (S = Q K^T)", cs);
  fa_sm103::mat::row_softmax_kernel<<<static_cast<unsigned>(BH * N), fa_sm103::mat::kRowThreads, 0,
                                      s>>>(S, P, l_round, lse, n, causal ? 1 : 0);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_error("row softmax launch", e);
  // column-major view: acc^T (d x N) = V^T (d x N) * P^T (N x N), i.e. acc[i] = sum_j P[i][j] v_j
  cs = cublasGemmStridedBatchedEx(h, CUBLAS_OP_N, CUBLAS_OP_N, dd, n, n, &one, v, CUDA_R_16BF, dd,
                                  sNd, P, CUDA_R_16BF, n, sN2, &zero, acc, CUDA_R_32F, dd, sNd,
                                  static_cast<int>(BH), CUBLAS_COMPUTE_32F, CUBLAS_GEMM_DEFAULT);
  if (cs != CUBLAS_STATUS_SUCCESS) return cublas_error("cublasGemmStridedBatchedEx (P V)", cs);
  const int64_t quads = BH * N * d / 4;
  fa_sm103::mat::normalise_kernel<<<static_cast<unsigned>((quads + 255) / 256), 256, 0, s>>>(
      reinterpret_cast<const float4*>(acc), l_round, static_cast<uint2*>(o), quads, dd);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_error("normalise launch", e);
  return FA_OK;
}

const char* fa_baseline_last_error(void) { return t_last_error.c_str(); }

}  // extern "C"
