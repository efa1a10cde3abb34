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
constexpr size_t kRecordBytes = 49664;  // operand record of one (64-token chunk, head)

static __device__ __align__(256) unsigned char g_build_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
void *g_scratch_ptr[kMaxDevices];
cudaError_t g_scratch_err[kMaxDevices];
std::once_flag g_scratch_once[kMaxDevices];

// Device address of the scratch array on the current device.  The host-side name
// g_build_scratch is only a stand-in, never a device address, so the address is
// looked up with cudaGetSymbolAddress once per device (with that device current).
cudaError_t scratch_ptr(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::call_once(g_scratch_once[dev], [dev]() {
    void *p = nullptr;
    g_scratch_err[dev] = cudaGetSymbolAddress(&p, g_build_scratch);
    g_scratch_ptr[dev] = p;
  });
  if (g_scratch_err[dev] != cudaSuccess) return g_scratch_err[dev];
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
  // Shapes whose build needs no workspace go straight through.
  if (hypic_build_workspace_bytes(shape, n_seg, max_len) == 0)
    return hypic_segment_build_batched(shape, n_seg, seg_bounds, max_len, n_tokens, k, v, q, alpha, beta, T_out,
                                       S_out, o_out, nullptr, 0, stream);
  // The build works through the heads in blocks that fit the scratch; one head's
  // records must fit, which bounds n_seg * ceil(max_len / 64).
  const size_t one_head = (size_t)n_seg * (size_t)((max_len + 63) / 64) * hypic::kRecordBytes;
  if (one_head > hypic::kScratchBytes) return HYPIC_ENOSPACE;
  void *scratch = nullptr;
  if (hypic::scratch_ptr(&scratch) != cudaSuccess) return HYPIC_ECUDA;
  return hypic_segment_build_batched(shape, n_seg, seg_bounds, max_len, n_tokens, k, v, q, alpha, beta, T_out,
                                     S_out, o_out, scratch, hypic::kScratchBytes, stream);
}
