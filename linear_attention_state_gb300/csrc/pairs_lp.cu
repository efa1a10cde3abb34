// 16-bit storage of cached pairs: rounds fp32 (T_C, S_{C|0}) to bf16 (round to nearest even).
// The paper sizes its cache with 16-bit T_C and S (HYPIC reading notes, Method 3, Table 3);
// composition then reads half the bytes per step (compose_tc.cu, chain.cu take bf16 pools).
#include <cuda_bf16.h>

#include "common.cuh"

namespace hypic {
namespace {

// Grid-stride over 8-element groups (16-byte stores); `n` is a multiple of 8 in the groups part,
// the tail is handled element by element.
__global__ void __launch_bounds__(256) round_bf16_kernel(const float *__restrict__ src,
                                                         __nv_bfloat16 *__restrict__ dst, int64_t n) {
  const int64_t groups = n / 8;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; g < groups; g += stride) {
    const float4 a = reinterpret_cast<const float4 *>(src)[2 * g];
    const float4 b = reinterpret_cast<const float4 *>(src)[2 * g + 1];
    const __nv_bfloat162 p0 = __floats2bfloat162_rn(a.x, a.y), p1 = __floats2bfloat162_rn(a.z, a.w);
    const __nv_bfloat162 p2 = __floats2bfloat162_rn(b.x, b.y), p3 = __floats2bfloat162_rn(b.z, b.w);
    uint4 o;
    o.x = *reinterpret_cast<const uint32_t *>(&p0);
    o.y = *reinterpret_cast<const uint32_t *>(&p1);
    o.z = *reinterpret_cast<const uint32_t *>(&p2);
    o.w = *reinterpret_cast<const uint32_t *>(&p3);
    reinterpret_cast<uint4 *>(dst)[g] = o;
  }
  for (int64_t i = groups * 8 + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
    dst[i] = __float2bfloat16_rn(src[i]);
}

cudaError_t round_bf16(const float *src, void *dst, int64_t n, int sms, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  const int64_t groups = (n + 7) / 8;
  int64_t blocks = (groups + 255) / 256;
  const int64_t cap = (int64_t)(sms > 0 ? sms : 152) * 8;
  if (blocks > cap) blocks = cap;
  round_bf16_kernel<<<(unsigned)blocks, 256, 0, st>>>(src, static_cast<__nv_bfloat16 *>(dst), n);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_pairs_to_bf16(const float *T, const float *S, void *T_lp, void *S_lp, int64_t t_elems,
                                 int64_t s_elems, cudaStream_t st) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaError_t e = round_bf16(T, T_lp, t_elems, sms, st);
  if (e != cudaSuccess) return e;
  return round_bf16(S, S_lp, s_elems, sms, st);
}

}  // namespace hypic
