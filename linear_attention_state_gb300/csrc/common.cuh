// Internal declarations shared by the libhypic translation units.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "hypic.h"

namespace hypic {

// Tensor-of-tokens view: element (tok, h, i) of k/q/v lives at (tok*H + h)*D + i.
struct TokenSrc {
  const void *k, *v, *q;
  const float *alpha, *beta;
  int in_dtype;  // HYPIC_F32 or HYPIC_BF16
};

// Records the first device-side error in the status word (never traps).
__device__ __forceinline__ void set_error(int *err, int code) {
  if (err) atomicCAS(err, 0, code);
}

template <typename Tin>
__device__ __forceinline__ float to_f32(Tin x);
template <>
__device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

// ---- launchers (host) -------------------------------------------------------------------

// Which rows of the token axis form segment s: bounds[2s], bounds[2s+1] if bounds is
// non-null, else [s*uni_stride + uni_offset, + uni_len).
struct SegMap {
  const int64_t *bounds;
  int64_t uni_stride, uni_offset, uni_len;
  int64_t max_len;   // a body longer than this is rejected (EDEVICE)
  int64_t n_tokens;  // token-axis extent (bounds check), < 0 = unchecked
};

struct RecurrentArgs {
  int H, D, fam;
  int n_seg;
  SegMap seg;
  TokenSrc src;
  const float *S_in;  // [n_seg, H, D, D] or null (zero)
  float *S_out;       // [n_seg, H, D, D]
  float *T_out;       // [n_seg, H, t_size] (build) or null (advance only)
  float *o_out;       // [tokens, H, D] or null
  int *err;
};
cudaError_t launch_recurrent(const RecurrentArgs &a, cudaStream_t st);

// Chunked tcgen05 build (d = 128, bf16 inputs, delta families, with or without per-token outputs).
// The workspace holds per-(chunk, head) operand records; the build runs over blocks
// of heads that fit in the workspace it is given (at least one head).
bool build_tc_supported(int D, int fam, int in_dtype, bool want_o);
size_t build_tc_workspace_bytes(int H, int n_seg, int64_t max_len, bool want_o);  // preferred size
size_t build_tc_min_workspace(int n_seg, int64_t max_len, bool want_o);          // one head
cudaError_t launch_build_tc(const RecurrentArgs &a, void *ws, size_t ws_bytes, cudaStream_t st);

// Chunked tcgen05 build for the KDA family (d = 128, bf16 inputs, no per-token outputs): per-(chunk,
// head) operand records in the workspace, processed over blocks of heads that fit.
bool build_kda_tc_supported(int D, int fam, int in_dtype, bool want_o);
size_t build_kda_tc_workspace_bytes(int H, int n_seg, int64_t max_len);  // preferred size
size_t build_kda_tc_min_workspace(int n_seg, int64_t max_len);           // one head
cudaError_t launch_build_kda_tc(const RecurrentArgs &a, void *ws, size_t ws_bytes, cudaStream_t st);

// Tensor-core build for the scalar and diagonal decay families (d = 128, bf16 inputs, no
// per-token outputs): one accumulating GEMM per (segment, head), no workspace.
bool build_decay_tc_supported(int D, int fam, int in_dtype, bool want_o);
cudaError_t launch_build_decay_tc(const RecurrentArgs &a, cudaStream_t st);

struct ChainArgs {
  int H, D, fam;
  int B, n, w;
  const int32_t *idx;  // [B, n] or null: step j of chain uses pool entry j
  int64_t pool_size;
  const void *pool_T;  // [P, H, t_size]  fp32, or bf16 when pair_bf16
  const void *pool_S;  // [P, H, D, D]     same element type
  int pair_bf16;
  const float *S_init;  // [B, H, D, D] or null
  float *S_out;         // final [B, H, D, D]
  // scan mode: record every prefix; T half of the augmented state goes to T_rec
  int scan;
  float *T_rec;  // [n, H, t_size]
  float *S_rec;  // [n, H, D, D]
  TokenSrc seam;  // seam tokens [B, n-1, w, H, D]
  float *o_out;   // [B, n-1, w, H, D] or null
  int *err;
  void *ws;         // scan: optional workspace for the two-level scan (null: one chain per head)
  size_t ws_bytes;
};
cudaError_t launch_chain(const ChainArgs &a, cudaStream_t st);

// tcgen05 composition chain (d = 128, delta families): compose, assemble and scan.
bool compose_tc_supported(int D, int fam);
cudaError_t launch_compose_tc(const ChainArgs &a, cudaStream_t st);
size_t scan_pipe32_workspace_bytes(int H, int n);  // two-level tensor-core scan (0: none used)

// fp32 pairs -> bf16 storage, round to nearest even (element counts; 16-byte aligned pointers).
cudaError_t launch_pairs_to_bf16(const float *T, const float *S, void *T_lp, void *S_lp, int64_t t_elems,
                                 int64_t s_elems, cudaStream_t st);

// Boundary patches (boundary.cu).
cudaError_t launch_rope_shift(const void *in, void *out, int64_t rows, int d, int r, double base, long long delta,
                              int dtype, int *err, cudaStream_t st);
cudaError_t launch_state_rerotate(float *S, int64_t mats, int dk, int dv, int r, double base, long long delta,
                                  int *err, cudaStream_t st);
cudaError_t launch_conv_tail(const void *x, int64_t n_tokens, int C, int k, int n_seg, const int64_t *bounds,
                             void *tail, int dtype, int *err, cudaStream_t st);
cudaError_t launch_conv_seam(const void *xs, const void *tail, const float *W, const float *bias, int B, int w, int C,
                             int k, int act, int dtype, float *y, cudaStream_t st);

// Bounded-wait self-test (see hypic_selftest_bounded_wait).
cudaError_t launch_bounded_wait_selftest(long long limit_cycles, int *err, cudaStream_t st);

}  // namespace hypic
