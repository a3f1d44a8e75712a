/*
 * fa_baseline.h -- C ABI of libfa_baseline.so, the materialised attention baseline.
 *
 * A library of its own: it links cuBLAS, which the tiled forward library (fa.h,
 * libfa_sm103.so) does not.  It computes the same result as fa_fwd the way the pages'
 * `standard_attention` does (aiml.sh "Speed up long contexts with FlashAttention",
 * lab.py), holding the N x N matrices in device memory, so the traffic and time the
 * tiled kernels avoid can be measured.  Status codes are fa.h's.
 */
#ifndef FA_BASELINE_H
#define FA_BASELINE_H

#include "fa.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * fa_fwd_materialised -- the materialised baseline: the same result computed the way the
 * pages' `standard_attention` does it (aiml.sh "Speed up long contexts with
 * FlashAttention", lab.py), with the N x N matrices in device memory:
 *     S = scale * Q K^T            fp32 [B*H, N, N] in the workspace (cuBLAS batched GEMM)
 *     P = exp(S - row max) + mask  bf16 [B*H, N, N] in the workspace, with the row sums
 *                                  of the rounded P and lse = ln sum_j exp(s_j) (this
 *                                  library's row kernel; masked entries are 0)
 *     acc = P V                    fp32 [B*H, N, d] in the workspace (cuBLAS batched GEMM)
 *     O = acc / row sum            bf16 (this library's kernel)
 * It exists to measure the traffic and time the tiled kernels avoid (the pages model
 * 4 H N^2 elements of such traffic per batch); it is not a fast path.
 *
 *   workspace  device memory, 256-byte aligned, caller-owned, at least
 *              fa_materialised_workspace_bytes(B, H, N, d) (about 6 B H N^2 + 4 B H N d
 *              bytes); must not overlap any tensor.  Its contents on entry do not matter.
 * Other arguments and errors as fa_fwd (N up to 2^20 and B*H*N < 2^31 here; error
 * details in fa_baseline_last_error()).  The first call on a device creates a cuBLAS
 * handle (cuBLAS allocates its own device workspace then); calls are serialised on a
 * library lock.
 */
int fa_fwd_materialised(const void* q, const void* k, const void* v, void* o, float* lse,
                        int64_t B, int64_t H, int64_t N, int64_t d, int causal, float scale,
                        void* workspace, size_t workspace_bytes, void* stream);

/* Workspace bytes fa_fwd_materialised needs (S, P, acc and row sums, each rounded up to a
   multiple of 256 bytes); -1 on bad or too large sizes or an unsupported head dim. */
int64_t fa_materialised_workspace_bytes(int64_t B, int64_t H, int64_t N, int64_t d);

/* Detail of the last error of this library on this host thread ("" after a success). */
const char* fa_baseline_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_BASELINE_H */
