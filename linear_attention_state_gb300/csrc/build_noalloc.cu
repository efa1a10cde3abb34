// Allocation-free variant of the batched segment build.
//
// Some callers cannot allocate device memory themselves: code embedded in a host
// framework that owns every device allocation through its own pool and exposes
// no allocator, or a serving process that runs with a fixed memory budget and
// must not allocate after start-up.  They cannot provide the workspace the
// tensor-core build needs.  This entry point uses a fixed scratch array that
// lives in the library itself (a file-scope __device__ array, so every GPU that
// loads the library holds it until the process exits) and otherwise runs the
// same build as hypic_segment_build_batched.
#include <mutex>

#include "common.cuh"

namespace hypic {
namespace {

constexpr size_t kScratchBytes = HYPIC_NOALLOC_SCRATCH_BYTES;  // per device

static __device__ __align__(256) unsigned char g_build_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
void *g_scratch_ptr[kMaxDevices];
std::mutex g_scratch_mu[kMaxDevices];

// Device address of the scratch array on the current device.  The host-side name
// g_build_scratch is only a stand-in, never a device address, so the address is
// looked up with cudaGetSymbolAddress (with the device current).  Only a successful
// lookup is kept: a failed one (say, a first call made while a stream is being
// captured) is tried again on the next call instead of failing every later call.
cudaError_t scratch_ptr(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu[dev]);
  if (!g_scratch_ptr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_build_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace hypic

extern "C" hypic_status hypic_segment_build_batched_noalloc(const hypic_shape *shape, int32_t n_seg,
                                                            const int64_t *seg_bounds, int64_t max_len,
                                                            int64_t n_tokens, const void *k, const void *v,
                                                            const void *q, const float *alpha, const float *beta,
                                                            float *T_out, float *S_out, float *o_out,
                                                            hypic_stream_t stream) {
  if (!shape || n_seg < 0 || max_len < 0) return HYPIC_EINVAL;
  // With per-token outputs (o_out given) the build keeps the larger record per (chunk, head).
  const bool want_o = o_out != nullptr;
  const size_t need = want_o ? hypic_build_workspace_bytes_outputs(shape, n_seg, max_len)
                             : hypic_build_workspace_bytes(shape, n_seg, max_len);
  // Shapes whose build needs no workspace go straight through.
  if (need == 0)
    return hypic_segment_build_batched(shape, n_seg, seg_bounds, max_len, n_tokens, k, v, q, alpha, beta, T_out,
                                       S_out, o_out, nullptr, 0, stream);
  // The build works through the heads in blocks that fit the scratch; one head's
  // records must fit, which bounds n_seg * ceil(max_len / 64).
  const size_t one_head = (shape->family == HYPIC_FAM_KDA && !want_o)
                              ? hypic::build_kda_tc_min_workspace(n_seg, max_len)
                              : hypic::build_tc_min_workspace(n_seg, max_len, want_o);
  if (one_head > hypic::kScratchBytes) return HYPIC_ENOSPACE;
  void *scratch = nullptr;
  if (hypic::scratch_ptr(&scratch) != cudaSuccess) return HYPIC_ECUDA;
  return hypic_segment_build_batched(shape, n_seg, seg_bounds, max_len, n_tokens, k, v, q, alpha, beta, T_out,
                                     S_out, o_out, scratch, hypic::kScratchBytes, stream);
}
