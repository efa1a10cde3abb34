// Chain kernels: compose, fused request assembly and the affine scan, fp32.
//
// Compose applies the cached pairs in prompt order, S <- T_C S + S_{C|0}
// (HYPIC reading notes, Method 2 and paper Eq. (6)); assembly first advances
// the running state through the w seam tokens of each inner segment
// (Method 5, seam windows), emitting o_i = q_i^T S_i; the scan records every
// prefix of the composition (T_i, S_i) o (T_{i-1}, S_{i-1}) o ...
//
// Dense families: one 256-thread block per (request, head) keeps the running
// d x d state in shared memory for the whole chain; each step is a register-
// tiled fp32 GEMM against T staged by cp.async (double buffered, so the next
// T streams in while this step computes), and the S_{C|0} addend is loaded to
// registers at the top of the step.  The scan runs the augmented state
// [T_p | S_p] as two blocks per head (the T half starts at I and has no
// addend).  Scalar and diagonal families: one thread per state column.
#include <cstdlib>
#include <cstring>

#include "common.cuh"

namespace hypic {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
  const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;\n" ::); }

__device__ __forceinline__ int64_t pool_entry(const ChainArgs &a, int b, int j) {
  int64_t p = a.idx ? (int64_t)a.idx[(size_t)b * a.n + j] : (int64_t)j;
  if (p < 0 || p >= a.pool_size) {
    set_error(a.err, HYPIC_EDEVICE);
    p = 0;
  }
  return p;
}

template <int D>
__device__ __forceinline__ void stage_T(float *dst, const float *src, int tid) {
  constexpr int chunks = D * D / 4;
  for (int c = tid; c < chunks; c += kThreads) cp_async16(dst + 4 * c, src + 4 * c);
}

// Seam advance on the shared-memory state for the dense families: the gate first (a scalar a_t,
// 1, or KDA's per-channel g_t), y = gate * x, then x = y + b (v_j - k . y) k.
template <int D, typename Tin>
__device__ void seam_dense(const ChainArgs &a, float *S, float *sk, float *sq, float *red,
                           float *sab, float *sg, int b, int j, int h) {
  constexpr int PARTS = kThreads / D;
  constexpr int RP = D / PARTS;
  const int tid = threadIdx.x, col = tid % D, part = tid / D;
  const Tin *K = static_cast<const Tin *>(a.seam.k);
  const Tin *V = static_cast<const Tin *>(a.seam.v);
  const Tin *Q = static_cast<const Tin *>(a.seam.q);
  const int H = a.H;
  for (int t = 0; t < a.w; ++t) {
    const size_t tok = ((size_t)b * (a.n - 1) + (j - 1)) * a.w + t;
    __syncthreads();
    if (tid < D) {
      const size_t g = (tok * H + h) * D + tid;
      sk[tid] = to_f32<Tin>(K[g]);
      sk[D + tid] = to_f32<Tin>(V[g]);
      if (a.o_out) sq[tid] = to_f32<Tin>(Q[g]);
      if (a.fam == HYPIC_FAM_KDA) sg[tid] = a.seam.alpha[g];
    }
    if (tid == 0) {
      sab[0] = a.fam == HYPIC_FAM_GATED_DELTA ? a.seam.alpha[tok * H + h] : 1.f;
      sab[1] = a.seam.beta[tok * H + h];
    }
    __syncthreads();
    const bool kda = a.fam == HYPIC_FAM_KDA;
    float c = 0.f;
#pragma unroll 8
    for (int r = 0; r < RP; ++r) {
      const int i = part * RP + r;
      const float y = (kda ? sg[i] : sab[0]) * S[i * D + col];
      S[i * D + col] = y;
      c = fmaf(sk[i], y, c);
    }
    red[part * D + col] = c;
    __syncthreads();
    c = 0.f;
#pragma unroll
    for (int p = 0; p < PARTS; ++p) c += red[p * D + col];
    const float coef = sab[1] * (sk[D + col] - c);
#pragma unroll 8
    for (int r = 0; r < RP; ++r) {
      const int i = part * RP + r;
      S[i * D + col] = fmaf(coef, sk[i], S[i * D + col]);
    }
    if (a.o_out) {
      __syncthreads();
      float o = 0.f;
#pragma unroll 8
      for (int r = 0; r < RP; ++r) {
        const int i = part * RP + r;
        o = fmaf(sq[i], S[i * D + col], o);
      }
      red[part * D + col] = o;
      __syncthreads();
      if (part == 0) {
        o = 0.f;
#pragma unroll
        for (int p = 0; p < PARTS; ++p) o += red[p * D + col];
        a.o_out[(tok * H + h) * D + col] = o;
      }
    }
  }
  __syncthreads();
}

template <int D, typename Tin>
__global__ void __launch_bounds__(kThreads, 1) chain_dense_kernel(ChainArgs a) {
  constexpr int TM = D / 16;  // thread tile TM x TM, 16 x 16 threads
  extern __shared__ __align__(16) float smem[];
  float *S = smem;
  float *Tb = S + D * D;       // 2 buffers
  float *sk = Tb + 2 * D * D;  // k then v (2D)
  float *sq = sk + 2 * D;
  float *red = sq + D;         // kThreads floats
  float *sab = red + kThreads;  // 2 floats
  float *sg = sab + 4;          // D floats: KDA seam gate

  const int nhalf = a.scan ? 2 : 1;
  const int half = blockIdx.x % nhalf;
  const int rest = blockIdx.x / nhalf;
  const int h = rest % a.H;
  const int b = rest / a.H;
  const bool isT = a.scan && half == 0;
  const int tid = threadIdx.x;
  const int i0 = (tid / 16) * TM, j0 = (tid % 16) * TM;
  const int H = a.H;
  const size_t DD = (size_t)D * D;

  for (int e = tid; e < D * D; e += kThreads) {
    float v0 = 0.f;
    if (isT) v0 = (e / D == e % D) ? 1.f : 0.f;
    else if (!a.scan && a.S_init) v0 = a.S_init[((size_t)b * H + h) * DD + e];
    S[e] = v0;
  }
  const float *poolT = static_cast<const float *>(a.pool_T), *poolS = static_cast<const float *>(a.pool_S);
  if (a.n > 0) stage_T<D>(Tb, poolT + ((size_t)pool_entry(a, b, 0) * H + h) * DD, tid);
  cp_async_commit();

  for (int j = 0; j < a.n; ++j) {
    const int64_t p = pool_entry(a, b, j);
    cp_async_wait_all();
    __syncthreads();
    if (j + 1 < a.n)
      stage_T<D>(Tb + ((j + 1) & 1) * DD, poolT + ((size_t)pool_entry(a, b, j + 1) * H + h) * DD, tid);
    cp_async_commit();

    float add[TM][TM];
    const float *S0 = poolS + ((size_t)p * H + h) * DD;
#pragma unroll
    for (int r = 0; r < TM; ++r) {
      if constexpr (TM % 4 == 0) {
#pragma unroll
        for (int c = 0; c < TM; c += 4) {
          float4 v4 = make_float4(0.f, 0.f, 0.f, 0.f);
          if (!isT) v4 = __ldg(reinterpret_cast<const float4 *>(S0 + (size_t)(i0 + r) * D + j0 + c));
          add[r][c] = v4.x;
          add[r][c + 1] = v4.y;
          add[r][c + 2] = v4.z;
          add[r][c + 3] = v4.w;
        }
      } else {
#pragma unroll
        for (int c = 0; c < TM; ++c) add[r][c] = isT ? 0.f : __ldg(S0 + (size_t)(i0 + r) * D + j0 + c);
      }
    }
    if (!a.scan && a.w > 0 && j >= 1) seam_dense<D, Tin>(a, S, sk, sq, red, sab, sg, b, j, h);

    const float *T = Tb + (j & 1) * DD;
    float acc[TM][TM];
#pragma unroll
    for (int r = 0; r < TM; ++r)
#pragma unroll
      for (int c = 0; c < TM; ++c) acc[r][c] = 0.f;
#pragma unroll 2
    for (int k4 = 0; k4 < D; k4 += 4) {
      float4 tv[TM];
#pragma unroll
      for (int r = 0; r < TM; ++r) tv[r] = *reinterpret_cast<const float4 *>(T + (i0 + r) * D + k4);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        float sv[TM];
        if constexpr (TM % 4 == 0) {
#pragma unroll
          for (int c = 0; c < TM; c += 4) {
            const float4 s4 = *reinterpret_cast<const float4 *>(S + (k4 + kk) * D + j0 + c);
            sv[c] = s4.x;
            sv[c + 1] = s4.y;
            sv[c + 2] = s4.z;
            sv[c + 3] = s4.w;
          }
        } else {
#pragma unroll
          for (int c = 0; c < TM; ++c) sv[c] = S[(k4 + kk) * D + j0 + c];
        }
#pragma unroll
        for (int r = 0; r < TM; ++r) {
          const float t = kk == 0 ? tv[r].x : kk == 1 ? tv[r].y : kk == 2 ? tv[r].z : tv[r].w;
#pragma unroll
          for (int c = 0; c < TM; ++c) acc[r][c] = fmaf(t, sv[c], acc[r][c]);
        }
      }
    }
    __syncthreads();
    float *rec = a.scan ? (isT ? a.T_rec : a.S_rec) + ((size_t)j * H + h) * DD : nullptr;
#pragma unroll
    for (int r = 0; r < TM; ++r) {
      if constexpr (TM % 4 == 0) {
#pragma unroll
        for (int c = 0; c < TM; c += 4) {
          float4 o = make_float4(acc[r][c] + add[r][c], acc[r][c + 1] + add[r][c + 1],
                                 acc[r][c + 2] + add[r][c + 2], acc[r][c + 3] + add[r][c + 3]);
          *reinterpret_cast<float4 *>(S + (i0 + r) * D + j0 + c) = o;
          if (rec) *reinterpret_cast<float4 *>(rec + (size_t)(i0 + r) * D + j0 + c) = o;
        }
      } else {
#pragma unroll
        for (int c = 0; c < TM; ++c) {
          const float o = acc[r][c] + add[r][c];
          S[(i0 + r) * D + j0 + c] = o;
          if (rec) rec[(size_t)(i0 + r) * D + j0 + c] = o;
        }
      }
    }
  }
  cp_async_wait_all();
  __syncthreads();
  if (!a.scan) {
    float *out = a.S_out + ((size_t)b * H + h) * DD;
    for (int e = tid * 4; e < D * D; e += kThreads * 4)
      *reinterpret_cast<float4 *>(out + e) = *reinterpret_cast<const float4 *>(S + e);
  }
}

// Scalar and diagonal families: column-per-thread chain, HBM-bound.  Pairs are fp32 or bf16 (Tp).
template <int D, typename Tin, typename Tp>
__global__ void __launch_bounds__(D >= 64 ? 64 : D) chain_diag_kernel(ChainArgs a) {
  constexpr int TPC = D >= 64 ? 64 : D;
  constexpr int NCB = D / TPC;
  __shared__ __align__(16) float st[D];
  __shared__ __align__(16) float sk[D];
  __shared__ __align__(16) float sq[D];
  __shared__ __align__(16) float sg[D];
  const int cb = blockIdx.x % NCB;
  const int rest = blockIdx.x / NCB;
  const int h = rest % a.H;
  const int b = rest / a.H;
  const int tid = threadIdx.x;
  const int j = cb * TPC + tid;
  const int H = a.H;
  const size_t DD = (size_t)D * D;
  const bool diag = a.fam == HYPIC_FAM_DIAG;
  const int ts = diag ? D : 1;
  const Tin *K = static_cast<const Tin *>(a.seam.k);
  const Tin *V = static_cast<const Tin *>(a.seam.v);
  const Tin *Q = static_cast<const Tin *>(a.seam.q);

  float x[D];
#pragma unroll
  for (int i = 0; i < D; ++i)
    x[i] = (!a.scan && a.S_init) ? a.S_init[((size_t)b * H + h) * DD + (size_t)i * D + j] : 0.f;
  float tp = 1.f;  // scan: running T prefix of channel j (diag) or the scalar

  for (int jj = 0; jj < a.n; ++jj) {
    const int64_t p = pool_entry(a, b, jj);
    if (!a.scan && a.w > 0 && jj >= 1) {
      for (int t = 0; t < a.w; ++t) {
        const size_t tok = ((size_t)b * (a.n - 1) + (jj - 1)) * a.w + t;
        __syncthreads();
        for (int i = tid; i < D; i += TPC) {
          const size_t g = (tok * H + h) * D + i;
          sk[i] = to_f32<Tin>(K[g]);
          if (a.o_out) sq[i] = to_f32<Tin>(Q[g]);
          sg[i] = diag ? a.seam.alpha[g] : (a.fam == HYPIC_FAM_SCALAR_CONST ? a.seam.alpha[h] : a.seam.alpha[tok * H + h]);
        }
        __syncthreads();
        const float vj = to_f32<Tin>(V[(tok * H + h) * D + j]);
        float o = 0.f;
#pragma unroll
        for (int i = 0; i < D; ++i) {
          x[i] = fmaf(sk[i], vj, sg[i] * x[i]);
          o = fmaf(sq[i], x[i], o);
        }
        if (a.o_out) a.o_out[(tok * H + h) * D + j] = o;
      }
    }
    __syncthreads();
    const Tp *Tq = static_cast<const Tp *>(a.pool_T) + ((size_t)p * H + h) * ts;
    for (int i = tid; i < D; i += TPC) st[i] = to_f32<Tp>(diag ? Tq[i] : Tq[0]);
    __syncthreads();
    const Tp *S0 = static_cast<const Tp *>(a.pool_S) + ((size_t)p * H + h) * DD;
#pragma unroll
    for (int i = 0; i < D; ++i) x[i] = fmaf(st[i], x[i], to_f32<Tp>(S0[(size_t)i * D + j]));
    if (a.scan) {
      tp *= st[diag ? j : 0];
      float *rec = a.S_rec + ((size_t)jj * H + h) * DD;
#pragma unroll
      for (int i = 0; i < D; ++i) rec[(size_t)i * D + j] = x[i];
      if (diag) a.T_rec[((size_t)jj * H + h) * D + j] = tp;
      else if (j == 0) a.T_rec[(size_t)jj * H + h] = tp;
    }
  }
  if (!a.scan) {
#pragma unroll
    for (int i = 0; i < D; ++i) a.S_out[((size_t)b * H + h) * DD + (size_t)i * D + j] = x[i];
  }
}

template <int D, typename Tin>
cudaError_t launch_d(const ChainArgs &a, cudaStream_t st) {
  const bool dense = a.fam == HYPIC_FAM_DELTA || a.fam == HYPIC_FAM_GATED_DELTA || a.fam == HYPIC_FAM_KDA;
  if (dense) {
    if (a.pair_bf16) return cudaErrorInvalidValue;  // rejected by the API before any launch
    const long long blocks = (long long)a.B * a.H * (a.scan ? 2 : 1);
    if (blocks <= 0) return cudaSuccess;
    const size_t smem = sizeof(float) * (3 * D * D + 3 * D + kThreads + 4 + D);
    cudaError_t e = cudaFuncSetAttribute(chain_dense_kernel<D, Tin>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    chain_dense_kernel<D, Tin><<<(unsigned)blocks, kThreads, smem, st>>>(a);
  } else {
    constexpr int TPC = D >= 64 ? 64 : D;
    const long long blocks = (long long)a.B * a.H * (D / TPC);
    if (blocks <= 0) return cudaSuccess;
    if (a.pair_bf16) chain_diag_kernel<D, Tin, __nv_bfloat16><<<(unsigned)blocks, TPC, 0, st>>>(a);
    else chain_diag_kernel<D, Tin, float><<<(unsigned)blocks, TPC, 0, st>>>(a);
  }
  return cudaGetLastError();
}

template <typename Tin>
cudaError_t launch_t(const ChainArgs &a, cudaStream_t st) {
  switch (a.D) {
    case 16: return launch_d<16, Tin>(a, st);
    case 32: return launch_d<32, Tin>(a, st);
    case 64: return launch_d<64, Tin>(a, st);
    case 128: return launch_d<128, Tin>(a, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

// HYPIC_COMPOSE_PATH=simt keeps the fp32 SIMT chain where the tensor-core chain applies
// (for comparisons); read at every call.
static bool force_simt() {
  const char *v = getenv("HYPIC_COMPOSE_PATH");
  return v && strcmp(v, "simt") == 0;
}

cudaError_t launch_chain(const ChainArgs &a, cudaStream_t st) {
  if (compose_tc_supported(a.D, a.fam) && !force_simt()) return launch_compose_tc(a, st);
  if (a.seam.in_dtype == HYPIC_BF16) return launch_t<__nv_bfloat16>(a, st);
  return launch_t<float>(a, st);
}

}  // namespace hypic
