// Boundary patches of the reuse path (HYPIC reading notes, Method part 6: causal convolution and
// RoPE at segment boundaries; paper Sec. 4.2-4.3, Eqs. (7), (8)).  All four are elementwise or
// nearly so and HBM-bound; each thread handles whole 16-bit or 32-bit elements along the
// contiguous axis so that a warp reads and writes full lines.
//
// * RoPE key shift, Eq. (8): K_b = R(b - a) K_a.  Rotate-half pairs (i, i + r/2), r = rotary
//   dims (the rest pass through), frequencies theta_i = base^(-2i/r), pair i turned by
//   D theta_i.  The angles are reduced modulo 2 pi in double precision before the cosine and
//   sine are taken, so a shift of 10^5 positions keeps full fp32 accuracy (a float product
//   D * theta_0 alone would be off by ~0.01 rad); each CTA builds the r/2-entry table once.
// * State re-rotation for the scalar families, Eq. (7): S_{C|b} = R(b - a) S_{C|a}, on the key
//   (row) index of S.
// * Causal conv tail: the last k - 1 inputs of each segment body, zero-padded in front.
// * Causal conv over the seam window: y_t = act(bias + sum_j W[c][j] x_{t-k+1+j}), with inputs
//   before the segment start taken from the previous segment's tail.
#include <cuda_bf16.h>

#include "common.cuh"

namespace hypic {
namespace {

constexpr int NT = 256;
constexpr int MAX_HALF = 256;  // r/2 <= 256 (r <= 512)

template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// cos/sin of D * base^(-2i/r) for i < r/2, reduced modulo 2 pi in double precision.
__device__ void rope_table(float *cs, float *sn, int half, int r, double base, long long delta) {
  const double two_pi = 6.283185307179586476925286766559;
  for (int i = threadIdx.x; i < half; i += blockDim.x) {
    const double theta = pow(base, -2.0 * (double)i / (double)r);
    double ang = (double)delta * theta;
    ang -= two_pi * rint(ang / two_pi);
    double s, c;
    sincos(ang, &s, &c);
    cs[i] = (float)c;
    sn[i] = (float)s;
  }
}

// 16-byte groups of one element type: 8 bf16 or 4 fp32.
template <typename T>
struct Vec {
  static constexpr int N = 16 / sizeof(T);
  uint4 raw;
  __device__ __forceinline__ float get(int i) const { return to_f32<T>(reinterpret_cast<const T *>(&raw)[i]); }
  __device__ __forceinline__ void set(int i, float x) { reinterpret_cast<T *>(&raw)[i] = from_f32<T>(x); }
};

// Vectorised form for rows whose rotated half and pass-through part are whole 16-byte groups
// (16-byte aligned rows): one thread turns N consecutive pairs.
template <typename T>
__global__ void __launch_bounds__(NT) rope_shift_vec_kernel(const T *__restrict__ in, T *__restrict__ out,
                                                            int64_t rows, int d, int r, double base, long long delta) {
  __shared__ float cs[MAX_HALF], sn[MAX_HALF];
  constexpr int N = Vec<T>::N;
  const int half = r / 2;
  rope_table(cs, sn, half, r, base, delta);
  __syncthreads();
  const int gpr = half / N + (in != out ? (d - r) / N : 0);  // 16-byte groups per row
  const int64_t total = rows * gpr;
  for (int64_t e = (int64_t)blockIdx.x * NT + threadIdx.x; e < total; e += (int64_t)gridDim.x * NT) {
    const int64_t row = e / gpr;
    const int g = (int)(e - row * gpr);
    const T *src = in + row * d;
    T *dst = out + row * d;
    if (g < half / N) {
      const int i0 = g * N;
      Vec<T> x, y;
      x.raw = *reinterpret_cast<const uint4 *>(src + i0);
      y.raw = *reinterpret_cast<const uint4 *>(src + i0 + half);
      Vec<T> xo, yo;
#pragma unroll
      for (int q = 0; q < N; ++q) {
        const float a = x.get(q), b = y.get(q), c = cs[i0 + q], sv = sn[i0 + q];
        xo.set(q, c * a - sv * b);
        yo.set(q, sv * a + c * b);
      }
      *reinterpret_cast<uint4 *>(dst + i0) = xo.raw;
      *reinterpret_cast<uint4 *>(dst + i0 + half) = yo.raw;
    } else {
      const int c0 = r + (g - half / N) * N;
      *reinterpret_cast<uint4 *>(dst + c0) = *reinterpret_cast<const uint4 *>(src + c0);
    }
  }
}

// Rows of length d (token x head); rotated pairs then the pass-through dims.
template <typename T>
__global__ void __launch_bounds__(NT) rope_shift_kernel(const T *__restrict__ in, T *__restrict__ out, int64_t rows,
                                                        int d, int r, double base, long long delta) {
  __shared__ float cs[MAX_HALF], sn[MAX_HALF];
  const int half = r / 2;
  rope_table(cs, sn, half, r, base, delta);
  __syncthreads();
  const int per_row = half + (in != out ? d - r : 0);
  const int64_t total = rows * per_row;
  for (int64_t e = (int64_t)blockIdx.x * NT + threadIdx.x; e < total; e += (int64_t)gridDim.x * NT) {
    const int64_t row = e / per_row;
    const int i = (int)(e - row * per_row);
    const T *src = in + row * d;
    T *dst = out + row * d;
    if (i < half) {
      const float x = to_f32<T>(src[i]), y = to_f32<T>(src[i + half]);
      dst[i] = from_f32<T>(cs[i] * x - sn[i] * y);
      dst[i + half] = from_f32<T>(sn[i] * x + cs[i] * y);
    } else {
      const int c = r + (i - half);
      dst[c] = src[c];
    }
  }
}

// S [mats, dk, dv] in place, 4 columns per thread (dv a multiple of 4).
__global__ void __launch_bounds__(NT) state_rerotate_vec_kernel(float *__restrict__ S, int64_t mats, int dk, int dv,
                                                                int r, double base, long long delta) {
  __shared__ float cs[MAX_HALF], sn[MAX_HALF];
  const int half = r / 2;
  rope_table(cs, sn, half, r, base, delta);
  __syncthreads();
  const int q4 = dv / 4;
  const int64_t per_mat = (int64_t)half * q4;
  const int64_t total = mats * per_mat;
  for (int64_t e = (int64_t)blockIdx.x * NT + threadIdx.x; e < total; e += (int64_t)gridDim.x * NT) {
    const int64_t m = e / per_mat;
    const int rem = (int)(e - m * per_mat);
    const int i = rem / q4, j = 4 * (rem - i * q4);
    float4 *px = reinterpret_cast<float4 *>(S + (m * dk + i) * dv + j);
    float4 *py = reinterpret_cast<float4 *>(S + (m * dk + i + half) * dv + j);
    const float4 x = *px, y = *py;
    const float c = cs[i], sv = sn[i];
    *px = make_float4(c * x.x - sv * y.x, c * x.y - sv * y.y, c * x.z - sv * y.z, c * x.w - sv * y.w);
    *py = make_float4(sv * x.x + c * y.x, sv * x.y + c * y.y, sv * x.z + c * y.z, sv * x.w + c * y.w);
  }
}

// S [mats, dk, dv] in place: rows i and i + r/2 (i < r/2) of each matrix.
__global__ void __launch_bounds__(NT) state_rerotate_kernel(float *__restrict__ S, int64_t mats, int dk, int dv,
                                                            int r, double base, long long delta) {
  __shared__ float cs[MAX_HALF], sn[MAX_HALF];
  const int half = r / 2;
  rope_table(cs, sn, half, r, base, delta);
  __syncthreads();
  const int64_t per_mat = (int64_t)half * dv;
  const int64_t total = mats * per_mat;
  for (int64_t e = (int64_t)blockIdx.x * NT + threadIdx.x; e < total; e += (int64_t)gridDim.x * NT) {
    const int64_t m = e / per_mat;
    const int64_t rem = e - m * per_mat;
    const int i = (int)(rem / dv), j = (int)(rem - (int64_t)i * dv);
    float *A = S + m * dk * dv;
    const float x = A[(int64_t)i * dv + j], y = A[(int64_t)(i + half) * dv + j];
    A[(int64_t)i * dv + j] = cs[i] * x - sn[i] * y;
    A[(int64_t)(i + half) * dv + j] = sn[i] * x + cs[i] * y;
  }
}

template <typename T>
__global__ void __launch_bounds__(NT) conv_tail_kernel(const T *__restrict__ x, int64_t n_tokens, int C, int k,
                                                       int n_seg, const int64_t *__restrict__ bounds,
                                                       T *__restrict__ tail, int *err) {
  const int km1 = k - 1;
  const int64_t total = (int64_t)n_seg * km1 * C;
  for (int64_t e = (int64_t)blockIdx.x * NT + threadIdx.x; e < total; e += (int64_t)gridDim.x * NT) {
    const int64_t s = e / ((int64_t)km1 * C);
    const int64_t rem = e - s * km1 * C;
    const int m = (int)(rem / C), c = (int)(rem - (int64_t)m * C);
    const int64_t beg = bounds[2 * s], end = bounds[2 * s + 1];
    T v = from_f32<T>(0.f);
    if (beg < 0 || end < beg || end > n_tokens) {
      set_error(err, HYPIC_EDEVICE);
    } else {
      const int64_t t = end - km1 + m;
      if (t >= beg) v = x[t * C + c];
    }
    tail[e] = v;
  }
}

template <typename T>
__global__ void __launch_bounds__(NT) conv_seam_kernel(const T *__restrict__ xs, const T *__restrict__ tail,
                                                       const float *__restrict__ W, const float *__restrict__ bias,
                                                       int B, int w, int C, int k, int act, float *__restrict__ y) {
  const int64_t total = (int64_t)B * w * C;
  for (int64_t e = (int64_t)blockIdx.x * NT + threadIdx.x; e < total; e += (int64_t)gridDim.x * NT) {
    const int64_t b = e / ((int64_t)w * C);
    const int64_t rem = e - b * w * C;
    const int t = (int)(rem / C), c = (int)(rem - (int64_t)t * C);
    float acc = bias ? bias[c] : 0.f;
    for (int j = 0; j < k; ++j) {
      const int src = t - k + 1 + j;  // position relative to the segment start
      const float xv = src >= 0 ? to_f32<T>(xs[(b * w + src) * C + c])
                                : to_f32<T>(tail[(b * (k - 1) + (k - 1 + src)) * C + c]);
      acc = fmaf(W[(int64_t)c * k + j], xv, acc);
    }
    if (act == HYPIC_ACT_SILU) acc = acc / (1.f + expf(-acc));
    y[e] = acc;
  }
}

unsigned grid_for(int64_t total) {
  int dev = 0, sms = 152;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int64_t g = (total + NT - 1) / NT;
  const int64_t cap = (int64_t)sms * 8;
  if (g > cap) g = cap;
  return (unsigned)(g < 1 ? 1 : g);
}

}  // namespace

cudaError_t launch_rope_shift(const void *in, void *out, int64_t rows, int d, int r, double base, long long delta,
                              int dtype, cudaStream_t st) {
  const int64_t total = rows * (r / 2 + (in != out ? d - r : 0));
  if (total <= 0) return cudaSuccess;
  const int n = dtype == HYPIC_BF16 ? 8 : 4;  // elements per 16-byte group
  const bool vec = (r / 2) % n == 0 && (d - r) % n == 0 && d % n == 0 &&
                   (reinterpret_cast<uintptr_t>(in) & 15) == 0 && (reinterpret_cast<uintptr_t>(out) & 15) == 0;
  if (vec) {
    const int64_t groups = rows * ((r / 2) / n + (in != out ? (d - r) / n : 0));
    if (dtype == HYPIC_BF16)
      rope_shift_vec_kernel<__nv_bfloat16><<<grid_for(groups), NT, 0, st>>>(
          static_cast<const __nv_bfloat16 *>(in), static_cast<__nv_bfloat16 *>(out), rows, d, r, base, delta);
    else
      rope_shift_vec_kernel<float><<<grid_for(groups), NT, 0, st>>>(static_cast<const float *>(in),
                                                                    static_cast<float *>(out), rows, d, r, base, delta);
    return cudaGetLastError();
  }
  if (dtype == HYPIC_BF16)
    rope_shift_kernel<__nv_bfloat16><<<grid_for(total), NT, 0, st>>>(
        static_cast<const __nv_bfloat16 *>(in), static_cast<__nv_bfloat16 *>(out), rows, d, r, base, delta);
  else
    rope_shift_kernel<float><<<grid_for(total), NT, 0, st>>>(static_cast<const float *>(in),
                                                             static_cast<float *>(out), rows, d, r, base, delta);
  return cudaGetLastError();
}

cudaError_t launch_state_rerotate(float *S, int64_t mats, int dk, int dv, int r, double base, long long delta,
                                  cudaStream_t st) {
  const int64_t total = mats * (r / 2) * dv;
  if (total <= 0) return cudaSuccess;
  if (dv % 4 == 0 && (reinterpret_cast<uintptr_t>(S) & 15) == 0) {
    state_rerotate_vec_kernel<<<grid_for(total / 4), NT, 0, st>>>(S, mats, dk, dv, r, base, delta);
    return cudaGetLastError();
  }
  state_rerotate_kernel<<<grid_for(total), NT, 0, st>>>(S, mats, dk, dv, r, base, delta);
  return cudaGetLastError();
}

cudaError_t launch_conv_tail(const void *x, int64_t n_tokens, int C, int k, int n_seg, const int64_t *bounds,
                             void *tail, int dtype, int *err, cudaStream_t st) {
  const int64_t total = (int64_t)n_seg * (k - 1) * C;
  if (total <= 0) return cudaSuccess;
  if (dtype == HYPIC_BF16)
    conv_tail_kernel<__nv_bfloat16><<<grid_for(total), NT, 0, st>>>(
        static_cast<const __nv_bfloat16 *>(x), n_tokens, C, k, n_seg, bounds, static_cast<__nv_bfloat16 *>(tail), err);
  else
    conv_tail_kernel<float><<<grid_for(total), NT, 0, st>>>(static_cast<const float *>(x), n_tokens, C, k, n_seg,
                                                            bounds, static_cast<float *>(tail), err);
  return cudaGetLastError();
}

cudaError_t launch_conv_seam(const void *xs, const void *tail, const float *W, const float *bias, int B, int w, int C,
                             int k, int act, int dtype, float *y, cudaStream_t st) {
  const int64_t total = (int64_t)B * w * C;
  if (total <= 0) return cudaSuccess;
  if (dtype == HYPIC_BF16)
    conv_seam_kernel<__nv_bfloat16><<<grid_for(total), NT, 0, st>>>(static_cast<const __nv_bfloat16 *>(xs),
                                                                    static_cast<const __nv_bfloat16 *>(tail), W, bias,
                                                                    B, w, C, k, act, y);
  else
    conv_seam_kernel<float><<<grid_for(total), NT, 0, st>>>(static_cast<const float *>(xs),
                                                            static_cast<const float *>(tail), W, bias, B, w, C, k,
                                                            act, y);
  return cudaGetLastError();
}

}  // namespace hypic
