// Boundary patches of the reuse path (HYPIC reading notes, Method part 6: causal convolution and
// RoPE at segment boundaries; paper Sec. 4.2-4.3, Eqs. (7), (8)).  All four are elementwise or
// nearly so and HBM-bound; each thread handles whole 16-bit or 32-bit elements along the
// contiguous axis so that a warp reads and writes full lines.
//
// * RoPE key shift, Eq. (8): K_b = R(b - a) K_a.  Rotate-half pairs (i, i + r/2), r = rotary
//   dims (the rest pass through), frequencies theta_i = base^(-2i/r), pair i turned by
//   D theta_i.  The angles are reduced modulo 2 pi in double precision before the cosine and
//   sine are taken, so a shift of 10^5 positions keeps full fp32 accuracy (a float product
//   D * theta_0 alone would be off by ~0.01 rad).  Double precision is slow on this GPU (about
//   one fused multiply-add per cycle per SM), so the rotation kernels run one CTA per SM: each
//   SM builds the r/2-entry table once and then streams its share of the rows, several 16-byte
//   groups per thread in flight.
// * State re-rotation for the scalar families, Eq. (7): S_{C|b} = R(b - a) S_{C|a}, on the key
//   (row) index of S.
// * Causal conv tail: the last k - 1 inputs of each segment body, zero-padded in front.
// * Causal conv over the seam window: y_t = act(bias + sum_j W[c][j] x_{t-k+1+j}), with inputs
//   before the segment start taken from the previous segment's tail.
#include <cuda_bf16.h>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace hypic {
namespace {

constexpr int NT = 256;
constexpr int MAX_HALF = 256;  // r/2 <= 256 (r <= 512)
constexpr int NTR = 512;       // rotation kernels: threads per CTA, one CTA per SM
constexpr int UNR = 4;         // 16-byte groups a thread of the rotation kernels has in flight
// Staged rotation kernels: blocks of whole rows (the RoPE shift) or whole matrices (the state
// re-rotation) land in a ring of shared-memory stages by bulk copies, several blocks ahead.
constexpr int NTS = 512;                // threads of a staged CTA (one CTA per SM)
constexpr uint32_t ROPE_STAGE = 32768;  // bytes of rows per stage (at least one row)
constexpr int ROPE_NS = 4;
constexpr int RR_NS = 3;                // state re-rotation: one matrix per stage
constexpr uint32_t STAGED_SMEM_CAP = 200 * 1024;

template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// cos/sin of D * base^(-2i/r) for i < r/2.  Double precision is kept to what fixes the angle:
// theta_1 = base^(-2/r) once per CTA, theta_i = theta_1^i by binary powers (a relative error
// below 2^-45 for i < 256), the product D theta_i and its reduction modulo 2 pi with a two-term
// 2 pi; the cosine and sine of the reduced angle (|x| <= pi) are then taken in fp32.  Called by
// every thread of the CTA (it holds a barrier).
__device__ void rope_table(float *cs, float *sn, int half, int r, double base, long long delta) {
  __shared__ double theta1;
  const double two_pi_hi = 6.283185307179586232, two_pi_lo = 2.4492935982947064e-16;
  if (threadIdx.x == 0) theta1 = pow(base, -2.0 / (double)r);
  __syncthreads();
  for (int i = threadIdx.x; i < half; i += blockDim.x) {
    double th = 1.0, p = theta1;
    for (int e = i; e != 0; e >>= 1) {
      if (e & 1) th *= p;
      p *= p;
    }
    double ang = (double)delta * th;
    const double k = rint(ang * (1.0 / two_pi_hi));
    ang = fma(-k, two_pi_hi, ang);
    ang = fma(-k, two_pi_lo, ang);
    float s, c;
    sincosf((float)ang, &s, &c);
    cs[i] = c;
    sn[i] = s;
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
// (16-byte aligned rows): one thread turns N consecutive pairs.  Each thread first loads its
// next UNR groups, then rotates and stores them.
template <typename T>
__global__ void __launch_bounds__(NTR) rope_shift_vec_kernel(const T *__restrict__ in, T *__restrict__ out,
                                                             int64_t rows, int d, int r, double base, long long delta) {
  __shared__ float cs[MAX_HALF], sn[MAX_HALF];
  constexpr int N = Vec<T>::N;
  const int half = r / 2, hg = half / N;
  rope_table(cs, sn, half, r, base, delta);
  __syncthreads();
  const int gpr = hg + (in != out ? (d - r) / N : 0);  // 16-byte groups per row
  const int64_t total = rows * gpr;
  const int64_t stride = (int64_t)gridDim.x * NTR;
  for (int64_t e0 = (int64_t)blockIdx.x * NTR + threadIdx.x; e0 < total; e0 += UNR * stride) {
    Vec<T> x[UNR], y[UNR];
    int64_t row[UNR];
    int grp[UNR];
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      const int64_t e = e0 + u * stride;
      row[u] = e / gpr;
      grp[u] = (int)(e - row[u] * gpr);
      y[u].raw = make_uint4(0u, 0u, 0u, 0u);
      if (e < total) {
        const T *src = in + row[u] * d;
        if (grp[u] < hg) {
          x[u].raw = *reinterpret_cast<const uint4 *>(src + grp[u] * N);
          y[u].raw = *reinterpret_cast<const uint4 *>(src + grp[u] * N + half);
        } else {
          x[u].raw = *reinterpret_cast<const uint4 *>(src + r + (grp[u] - hg) * N);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      if (e0 + u * stride >= total) continue;
      T *dst = out + row[u] * d;
      if (grp[u] < hg) {
        const int i0 = grp[u] * N;
        Vec<T> xo, yo;
#pragma unroll
        for (int q = 0; q < N; ++q) {
          const float a = x[u].get(q), b = y[u].get(q), c = cs[i0 + q], sv = sn[i0 + q];
          xo.set(q, c * a - sv * b);
          yo.set(q, sv * a + c * b);
        }
        *reinterpret_cast<uint4 *>(dst + i0) = xo.raw;
        *reinterpret_cast<uint4 *>(dst + i0 + half) = yo.raw;
      } else {
        *reinterpret_cast<uint4 *>(dst + r + (grp[u] - hg) * N) = x[u].raw;
      }
    }
  }
}

// Waits (bounded) until stage `st` holds its block; every thread learns the outcome.
__device__ __forceinline__ bool stage_ready(uint64_t *bar, uint32_t parity, int *err) {
  int got = 1;
  if ((threadIdx.x & 31) == 0) got = tc::mbar_wait_cycles(bar, parity, err) ? 1 : 0;
  __syncwarp();
  return __shfl_sync(0xffffffffu, got, 0) != 0;
}

// Staged RoPE shift (16-byte-group rows, 16-byte-aligned tensors).  CTA b takes row blocks
// b, b + G, b + 2G, ... of `tile_rows` rows; thread 0 keeps ROPE_NS blocks in flight.  In place
// is safe: a block is read into shared memory before any of its rows is written.
template <typename T>
__global__ void __launch_bounds__(NTS) rope_shift_staged_kernel(const T *__restrict__ in, T *__restrict__ out,
                                                                int64_t rows, int d, int r, double base,
                                                                long long delta, int tile_rows, int *err) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(16) float cs[MAX_HALF];  // read as float4
  __shared__ __align__(16) float sn[MAX_HALF];
  __shared__ uint64_t full[ROPE_NS];
  __shared__ int abort_flag;
  constexpr int N = Vec<T>::N;
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 15) & ~uintptr_t(15));
  const int tid = threadIdx.x;
  const int half = r / 2, hg = half / N;
  const int gpr = hg + (in != out ? (d - r) / N : 0);
  const uint32_t row_bytes = (uint32_t)d * sizeof(T), stage_bytes = (uint32_t)tile_rows * row_bytes;
  const int64_t n_tiles = (rows + tile_rows - 1) / tile_rows;
  auto issue = [&](int64_t tile, int st) {
    const int64_t r0 = tile * tile_rows;
    const int nr = (int)(rows - r0 < tile_rows ? rows - r0 : tile_rows);
    tc::mbar_arrive_expect_tx(&full[st], (uint32_t)nr * row_bytes);
    tc::bulk_load(sm + st * stage_bytes, in + r0 * d, (uint32_t)nr * row_bytes, &full[st]);
  };
  if (tid == 0) {
    for (int q = 0; q < ROPE_NS; ++q) tc::mbar_init(&full[q], 1);
    tc::mbar_fence_init();
    abort_flag = 0;
    for (int q = 0; q < ROPE_NS; ++q)
      if (blockIdx.x + (int64_t)q * gridDim.x < n_tiles) issue(blockIdx.x + (int64_t)q * gridDim.x, q);
  }
  rope_table(cs, sn, half, r, base, delta);
  __syncthreads();
  int64_t k = 0;
  for (;; ++k) {
    const int64_t tile = blockIdx.x + k * gridDim.x;
    if (tile >= n_tiles) break;
    const int st = (int)(k % ROPE_NS);
    if (!stage_ready(&full[st], (uint32_t)(k / ROPE_NS) & 1u, err)) abort_flag = 1;
    const int64_t r0 = tile * tile_rows;
    const int nr = (int)(rows - r0 < tile_rows ? rows - r0 : tile_rows);
    const T *blk = reinterpret_cast<const T *>(sm + st * stage_bytes);
    if (!abort_flag) {
      for (int e = tid; e < nr * gpr; e += NTS) {
        const int row = e / gpr, g = e - row * gpr;
        const T *src = blk + (size_t)row * d;
        T *dst = out + (r0 + row) * d;
        if (g < hg) {
          const int i0 = g * N;
          Vec<T> x, y, xo, yo;
          x.raw = *reinterpret_cast<const uint4 *>(src + i0);
          y.raw = *reinterpret_cast<const uint4 *>(src + i0 + half);
#pragma unroll
          for (int q = 0; q < N; q += 4) {
            const float4 c4 = *reinterpret_cast<const float4 *>(cs + i0 + q);
            const float4 s4 = *reinterpret_cast<const float4 *>(sn + i0 + q);
            const float c[4] = {c4.x, c4.y, c4.z, c4.w}, sv[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const float a = x.get(q + u), b = y.get(q + u);
              xo.set(q + u, c[u] * a - sv[u] * b);
              yo.set(q + u, sv[u] * a + c[u] * b);
            }
          }
          *reinterpret_cast<uint4 *>(dst + i0) = xo.raw;
          *reinterpret_cast<uint4 *>(dst + i0 + half) = yo.raw;
        } else {
          const int c0 = r + (g - hg) * N;
          *reinterpret_cast<uint4 *>(dst + c0) = *reinterpret_cast<const uint4 *>(src + c0);
        }
      }
    }
    __syncthreads();  // the stage is consumed
    if (abort_flag) break;
    if (tid == 0 && tile + (int64_t)ROPE_NS * gridDim.x < n_tiles) issue(tile + (int64_t)ROPE_NS * gridDim.x, st);
  }
  if (abort_flag && tid == 0) {
    // Drain the blocks still in flight (bounded) before the CTA's shared memory is released.
    for (int64_t j = k; j < k + ROPE_NS && blockIdx.x + j * gridDim.x < n_tiles; ++j)
      tc::mbar_wait_cycles(&full[j % ROPE_NS], (uint32_t)(j / ROPE_NS) & 1u, nullptr, 200000000LL);
  }
}

// Staged state re-rotation: one [dk][dv] fp32 matrix per stage (dv a multiple of 4), in place.
__global__ void __launch_bounds__(NTS) state_rerotate_staged_kernel(float *__restrict__ S, int64_t mats, int dk,
                                                                    int dv, int r, double base, long long delta,
                                                                    int *err) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ float cs[MAX_HALF], sn[MAX_HALF];
  __shared__ uint64_t full[RR_NS];
  __shared__ int abort_flag;
  float *sm = reinterpret_cast<float *>((reinterpret_cast<uintptr_t>(smem_raw) + 15) & ~uintptr_t(15));
  const int tid = threadIdx.x;
  const int half = r / 2, q4 = dv / 4;
  const uint32_t mat_bytes = (uint32_t)dk * dv * 4u;
  auto issue = [&](int64_t m, int st) {
    tc::mbar_arrive_expect_tx(&full[st], mat_bytes);
    tc::bulk_load(sm + (size_t)st * dk * dv, S + m * dk * dv, mat_bytes, &full[st]);
  };
  if (tid == 0) {
    for (int q = 0; q < RR_NS; ++q) tc::mbar_init(&full[q], 1);
    tc::mbar_fence_init();
    abort_flag = 0;
    for (int q = 0; q < RR_NS; ++q)
      if (blockIdx.x + (int64_t)q * gridDim.x < mats) issue(blockIdx.x + (int64_t)q * gridDim.x, q);
  }
  rope_table(cs, sn, half, r, base, delta);
  __syncthreads();
  int64_t k = 0;
  for (;; ++k) {
    const int64_t m = blockIdx.x + k * gridDim.x;
    if (m >= mats) break;
    const int st = (int)(k % RR_NS);
    if (!stage_ready(&full[st], (uint32_t)(k / RR_NS) & 1u, err)) abort_flag = 1;
    const float *blk = sm + (size_t)st * dk * dv;
    float *A = S + m * dk * dv;
    if (!abort_flag) {
      for (int e = tid; e < half * q4; e += NTS) {
        const int i = e / q4, j = 4 * (e - i * q4);
        const float4 x = *reinterpret_cast<const float4 *>(blk + i * dv + j);
        const float4 y = *reinterpret_cast<const float4 *>(blk + (i + half) * dv + j);
        const float c = cs[i], sv = sn[i];
        *reinterpret_cast<float4 *>(A + (int64_t)i * dv + j) =
            make_float4(c * x.x - sv * y.x, c * x.y - sv * y.y, c * x.z - sv * y.z, c * x.w - sv * y.w);
        *reinterpret_cast<float4 *>(A + (int64_t)(i + half) * dv + j) =
            make_float4(sv * x.x + c * y.x, sv * x.y + c * y.y, sv * x.z + c * y.z, sv * x.w + c * y.w);
      }
    }
    __syncthreads();  // the stage is consumed
    if (abort_flag) break;
    if (tid == 0 && m + (int64_t)RR_NS * gridDim.x < mats) issue(m + (int64_t)RR_NS * gridDim.x, st);
  }
  if (abort_flag && tid == 0) {
    for (int64_t j = k; j < k + RR_NS && blockIdx.x + j * gridDim.x < mats; ++j)
      tc::mbar_wait_cycles(&full[j % RR_NS], (uint32_t)(j / RR_NS) & 1u, nullptr, 200000000LL);
  }
}

// Rows of length d (token x head); rotated pairs then the pass-through dims.
template <typename T>
__global__ void __launch_bounds__(NTR) rope_shift_kernel(const T *__restrict__ in, T *__restrict__ out, int64_t rows,
                                                        int d, int r, double base, long long delta) {
  __shared__ float cs[MAX_HALF], sn[MAX_HALF];
  const int half = r / 2;
  rope_table(cs, sn, half, r, base, delta);
  __syncthreads();
  const int per_row = half + (in != out ? d - r : 0);
  const int64_t total = rows * per_row;
  for (int64_t e = (int64_t)blockIdx.x * NTR + threadIdx.x; e < total; e += (int64_t)gridDim.x * NTR) {
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

// S [mats, dk, dv] in place, 4 columns per thread (dv a multiple of 4), UNR groups in flight.
__global__ void __launch_bounds__(NTR) state_rerotate_vec_kernel(float *__restrict__ S, int64_t mats, int dk, int dv,
                                                                 int r, double base, long long delta) {
  __shared__ float cs[MAX_HALF], sn[MAX_HALF];
  const int half = r / 2;
  rope_table(cs, sn, half, r, base, delta);
  __syncthreads();
  const int q4 = dv / 4;
  const int64_t per_mat = (int64_t)half * q4;
  const int64_t total = mats * per_mat;
  const int64_t stride = (int64_t)gridDim.x * NTR;
  for (int64_t e0 = (int64_t)blockIdx.x * NTR + threadIdx.x; e0 < total; e0 += UNR * stride) {
    float4 x[UNR], y[UNR];
    float *px[UNR];
    int row[UNR];
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      const int64_t e = e0 + u * stride;
      const int64_t m = e / per_mat;
      const int rem = (int)(e - m * per_mat);
      const int i = rem / q4, j = 4 * (rem - i * q4);
      row[u] = i;
      px[u] = S + (m * dk + i) * dv + j;
      if (e < total) {
        x[u] = *reinterpret_cast<const float4 *>(px[u]);
        y[u] = *reinterpret_cast<const float4 *>(px[u] + (int64_t)half * dv);
      }
    }
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      if (e0 + u * stride >= total) continue;
      const float c = cs[row[u]], sv = sn[row[u]];
      const float4 a = x[u], b = y[u];
      *reinterpret_cast<float4 *>(px[u]) =
          make_float4(c * a.x - sv * b.x, c * a.y - sv * b.y, c * a.z - sv * b.z, c * a.w - sv * b.w);
      *reinterpret_cast<float4 *>(px[u] + (int64_t)half * dv) =
          make_float4(sv * a.x + c * b.x, sv * a.y + c * b.y, sv * a.z + c * b.z, sv * a.w + c * b.w);
    }
  }
}

// S [mats, dk, dv] in place: rows i and i + r/2 (i < r/2) of each matrix.
__global__ void __launch_bounds__(NTR) state_rerotate_kernel(float *__restrict__ S, int64_t mats, int dk, int dv,
                                                             int r, double base, long long delta) {
  __shared__ float cs[MAX_HALF], sn[MAX_HALF];
  const int half = r / 2;
  rope_table(cs, sn, half, r, base, delta);
  __syncthreads();
  const int64_t per_mat = (int64_t)half * dv;
  const int64_t total = mats * per_mat;
  for (int64_t e = (int64_t)blockIdx.x * NTR + threadIdx.x; e < total; e += (int64_t)gridDim.x * NTR) {
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

// Rotation kernels: at most one CTA per SM, so the double-precision table is built once per SM.
unsigned grid_rot(int64_t items) {
  int dev = 0, sms = 152;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int64_t g = (items + NTR - 1) / NTR;
  if (g > sms) g = sms;
  return (unsigned)(g < 1 ? 1 : g);
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

template <typename T>
cudaError_t rope_staged(const void *in, void *out, int64_t rows, int d, int r, double base, long long delta,
                        int *err, cudaStream_t st) {
  const uint32_t row_bytes = (uint32_t)d * sizeof(T);
  const int tile_rows = (int)(ROPE_STAGE / row_bytes);
  const uint32_t smem = ROPE_NS * (uint32_t)tile_rows * row_bytes + 16;
  cudaError_t e = cudaFuncSetAttribute(rope_shift_staged_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  const int64_t tiles = (rows + tile_rows - 1) / tile_rows;
  rope_shift_staged_kernel<T><<<grid_rot(tiles * NTR), NTS, smem, st>>>(static_cast<const T *>(in),
                                                                         static_cast<T *>(out), rows, d, r, base,
                                                                         delta, tile_rows, err);
  return cudaGetLastError();
}

cudaError_t launch_rope_shift(const void *in, void *out, int64_t rows, int d, int r, double base, long long delta,
                              int dtype, int *err, cudaStream_t st) {
  const int64_t total = rows * (r / 2 + (in != out ? d - r : 0));
  if (total <= 0) return cudaSuccess;
  const int n = dtype == HYPIC_BF16 ? 8 : 4;  // elements per 16-byte group
  const bool vec = (r / 2) % n == 0 && (d - r) % n == 0 && d % n == 0 &&
                   (reinterpret_cast<uintptr_t>(in) & 15) == 0 && (reinterpret_cast<uintptr_t>(out) & 15) == 0;
  const uint32_t row_bytes = (uint32_t)d * (dtype == HYPIC_BF16 ? 2u : 4u);
  if (vec && row_bytes <= ROPE_STAGE) {
    return dtype == HYPIC_BF16 ? rope_staged<__nv_bfloat16>(in, out, rows, d, r, base, delta, err, st)
                               : rope_staged<float>(in, out, rows, d, r, base, delta, err, st);
  }
  if (vec) {
    const int64_t groups = rows * ((r / 2) / n + (in != out ? (d - r) / n : 0));
    if (dtype == HYPIC_BF16)
      rope_shift_vec_kernel<__nv_bfloat16><<<grid_rot(groups), NTR, 0, st>>>(
          static_cast<const __nv_bfloat16 *>(in), static_cast<__nv_bfloat16 *>(out), rows, d, r, base, delta);
    else
      rope_shift_vec_kernel<float><<<grid_rot(groups), NTR, 0, st>>>(static_cast<const float *>(in),
                                                                    static_cast<float *>(out), rows, d, r, base, delta);
    return cudaGetLastError();
  }
  if (dtype == HYPIC_BF16)
    rope_shift_kernel<__nv_bfloat16><<<grid_rot(total), NTR, 0, st>>>(
        static_cast<const __nv_bfloat16 *>(in), static_cast<__nv_bfloat16 *>(out), rows, d, r, base, delta);
  else
    rope_shift_kernel<float><<<grid_rot(total), NTR, 0, st>>>(static_cast<const float *>(in),
                                                             static_cast<float *>(out), rows, d, r, base, delta);
  return cudaGetLastError();
}

cudaError_t launch_state_rerotate(float *S, int64_t mats, int dk, int dv, int r, double base, long long delta,
                                  int *err, cudaStream_t st) {
  const int64_t total = mats * (r / 2) * dv;
  if (total <= 0) return cudaSuccess;
  const bool vec = dv % 4 == 0 && (reinterpret_cast<uintptr_t>(S) & 15) == 0;
  const uint32_t mat_bytes = (uint32_t)dk * dv * 4u;
  if (vec && RR_NS * mat_bytes + 16 <= STAGED_SMEM_CAP) {
    const uint32_t smem = RR_NS * mat_bytes + 16;
    cudaError_t e = cudaFuncSetAttribute(state_rerotate_staged_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    state_rerotate_staged_kernel<<<grid_rot(mats * NTR), NTS, smem, st>>>(S, mats, dk, dv, r, base, delta, err);
    return cudaGetLastError();
  }
  if (vec) {
    state_rerotate_vec_kernel<<<grid_rot(total / 4), NTR, 0, st>>>(S, mats, dk, dv, r, base, delta);
    return cudaGetLastError();
  }
  state_rerotate_kernel<<<grid_rot(total), NTR, 0, st>>>(S, mats, dk, dv, r, base, delta);
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
