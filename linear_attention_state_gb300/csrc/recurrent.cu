// Token-by-token recurrence kernels: the direct form of S_i = T_i S_{i-1} + u_i,
// o_i = q_i^T S_i (HYPIC reading notes, paper Eq. (2); variants of paper Table 1).
//
// Each column of the state evolves on its own: for the delta families
//   x <- a (x - b k (k . x)) + b v_j k   =   a x + b (v_j - a (k . x)) k,
// and for KDA (T = (I - b k k^T) diag(g)) y = g * x, x <- y + b (v_j - k . y) k,
// so one thread owns one column of the state in registers and the k, q vectors
// of a tile of tokens are staged in shared memory and read as broadcasts.  The
// build runs over the augmented state [T | S] (d_k x (d_k + d_v)) from [I | 0]:
// its T columns give T_C (the "S_0 = I, u = 0" pass of the two-pass build,
// paper Sec. 5) and its S columns give S_{C|0} in the same pass.  With a given
// initial state and S columns only, the same kernel is the seam advance.
//
// This kernel is the reference GPU path: every family, fp32 or bf16 inputs,
// d in {16, 32, 64, 128}.  The d = 128 delta build has a tensor-core path too.
#include "common.cuh"

namespace hypic {
namespace {

enum Kind { KIND_SCALAR = 0, KIND_DIAG = 1, KIND_DELTA = 2, KIND_KDA = 3 };

constexpr int kTile = 16;  // tokens staged per shared-memory tile

__device__ __forceinline__ void seg_range(const SegMap &m, int s, int64_t &b, int64_t &e, bool &ok) {
  if (m.bounds) {
    b = m.bounds[2 * s];
    e = m.bounds[2 * s + 1];
  } else {
    b = (int64_t)s * m.uni_stride + m.uni_offset;
    e = b + m.uni_len;
  }
  ok = (b >= 0) && (e >= b) && (e - b <= m.max_len) && (m.n_tokens < 0 || e <= m.n_tokens);
}

template <int D, int KIND, typename Tin>
__global__ void __launch_bounds__(D >= 64 ? 64 : D) recurrent_kernel(RecurrentArgs a) {
  constexpr int TPC = D >= 64 ? 64 : D;  // columns (threads) per block
  const bool build = a.T_out != nullptr;
  const bool dense_build = build && (KIND == KIND_DELTA || KIND == KIND_KDA);
  constexpr bool CHANNEL_GATE = KIND == KIND_DIAG || KIND == KIND_KDA;
  const int ncols = dense_build ? 2 * D : D;
  const int ncb = ncols / TPC;
  const int cb = blockIdx.x % ncb;
  const int rest = blockIdx.x / ncb;
  const int h = rest % a.H;
  const int s = rest / a.H;
  const int H = a.H;
  const int tid = threadIdx.x;
  const int j = cb * TPC + tid;             // column of the (augmented) state
  const bool isT = dense_build && j < D;    // uniform over the block
  const int jS = dense_build ? j - D : j;   // column of S when !isT

  int64_t beg, end;
  bool ok;
  seg_range(a.seg, s, beg, end, ok);
  if (!ok) {
    if (tid == 0 && cb == 0) set_error(a.err, HYPIC_EDEVICE);
    return;
  }
  const int64_t len = end - beg;

  __shared__ __align__(16) float sk[kTile][D];
  __shared__ __align__(16) float sq[kTile][D];
  __shared__ __align__(16) float sg[kTile][CHANNEL_GATE ? D : 1];
  __shared__ float sa[kTile], sb[kTile];

  const Tin *K = static_cast<const Tin *>(a.src.k);
  const Tin *V = static_cast<const Tin *>(a.src.v);
  const Tin *Q = static_cast<const Tin *>(a.src.q);
  const bool want_o = (a.o_out != nullptr) && !isT;
  const int fam = a.fam;

  float x[D];
  const size_t sidx = ((size_t)s * H + h) * D;  // row base of this (segment, head)
#pragma unroll
  for (int i = 0; i < D; ++i) {
    if (isT) x[i] = (i == j) ? 1.f : 0.f;
    else x[i] = a.S_in ? a.S_in[(sidx + i) * D + jS] : 0.f;
  }
  float tprod = 1.f;  // scalar / diagonal T_C: product of gates

  for (int64_t t0 = 0; t0 < len; t0 += kTile) {
    const int nt = (len - t0 < kTile) ? (int)(len - t0) : kTile;
    __syncthreads();
    for (int e = tid; e < nt * D; e += TPC) {
      const int t = e / D, i = e % D;
      const size_t g = ((size_t)(beg + t0 + t) * H + h) * D + i;
      sk[t][i] = to_f32<Tin>(K[g]);
      if (want_o) sq[t][i] = to_f32<Tin>(Q[g]);
      if (CHANNEL_GATE) sg[t][i] = a.src.alpha[g];
    }
    for (int t = tid; t < nt; t += TPC) {
      const size_t g = (size_t)(beg + t0 + t) * H + h;
      float av = 1.f, bv = 1.f;
      if (fam == HYPIC_FAM_SCALAR_CONST) av = a.src.alpha[h];
      else if (fam == HYPIC_FAM_SCALAR || fam == HYPIC_FAM_GATED_DELTA) av = a.src.alpha[g];
      if (fam == HYPIC_FAM_DELTA || fam == HYPIC_FAM_GATED_DELTA || fam == HYPIC_FAM_KDA) bv = a.src.beta[g];
      sa[t] = av;
      sb[t] = bv;
    }
    __syncthreads();
    for (int t = 0; t < nt; ++t) {
      const int64_t tok = beg + t0 + t;
      const float vj = isT ? 0.f : to_f32<Tin>(V[((size_t)tok * H + h) * D + jS]);
      const float at = sa[t];
      const float4 *k4 = reinterpret_cast<const float4 *>(sk[t]);
      if (KIND == KIND_DELTA) {
        float c0 = 0.f, c1 = 0.f, c2 = 0.f, c3 = 0.f;
#pragma unroll
        for (int i = 0; i < D / 4; ++i) {
          const float4 kv = k4[i];
          c0 = fmaf(kv.x, x[4 * i + 0], c0);
          c1 = fmaf(kv.y, x[4 * i + 1], c1);
          c2 = fmaf(kv.z, x[4 * i + 2], c2);
          c3 = fmaf(kv.w, x[4 * i + 3], c3);
        }
        const float c = (c0 + c1) + (c2 + c3);
        const float coef = sb[t] * (vj - at * c);
#pragma unroll
        for (int i = 0; i < D / 4; ++i) {
          const float4 kv = k4[i];
          x[4 * i + 0] = fmaf(coef, kv.x, at * x[4 * i + 0]);
          x[4 * i + 1] = fmaf(coef, kv.y, at * x[4 * i + 1]);
          x[4 * i + 2] = fmaf(coef, kv.z, at * x[4 * i + 2]);
          x[4 * i + 3] = fmaf(coef, kv.w, at * x[4 * i + 3]);
        }
      } else if (KIND == KIND_KDA) {
        const float4 *g4 = reinterpret_cast<const float4 *>(sg[t]);
        float c0 = 0.f, c1 = 0.f, c2 = 0.f, c3 = 0.f;
#pragma unroll
        for (int i = 0; i < D / 4; ++i) {
          const float4 kv = k4[i];
          const float4 gv = g4[i];
          x[4 * i + 0] *= gv.x;
          x[4 * i + 1] *= gv.y;
          x[4 * i + 2] *= gv.z;
          x[4 * i + 3] *= gv.w;
          c0 = fmaf(kv.x, x[4 * i + 0], c0);
          c1 = fmaf(kv.y, x[4 * i + 1], c1);
          c2 = fmaf(kv.z, x[4 * i + 2], c2);
          c3 = fmaf(kv.w, x[4 * i + 3], c3);
        }
        const float coef = sb[t] * (vj - ((c0 + c1) + (c2 + c3)));
#pragma unroll
        for (int i = 0; i < D / 4; ++i) {
          const float4 kv = k4[i];
          x[4 * i + 0] = fmaf(coef, kv.x, x[4 * i + 0]);
          x[4 * i + 1] = fmaf(coef, kv.y, x[4 * i + 1]);
          x[4 * i + 2] = fmaf(coef, kv.z, x[4 * i + 2]);
          x[4 * i + 3] = fmaf(coef, kv.w, x[4 * i + 3]);
        }
      } else if (KIND == KIND_SCALAR) {
#pragma unroll
        for (int i = 0; i < D / 4; ++i) {
          const float4 kv = k4[i];
          x[4 * i + 0] = fmaf(kv.x, vj, at * x[4 * i + 0]);
          x[4 * i + 1] = fmaf(kv.y, vj, at * x[4 * i + 1]);
          x[4 * i + 2] = fmaf(kv.z, vj, at * x[4 * i + 2]);
          x[4 * i + 3] = fmaf(kv.w, vj, at * x[4 * i + 3]);
        }
        tprod *= at;
      } else {  // KIND_DIAG
        const float4 *g4 = reinterpret_cast<const float4 *>(sg[t]);
#pragma unroll
        for (int i = 0; i < D / 4; ++i) {
          const float4 kv = k4[i];
          const float4 gv = g4[i];
          x[4 * i + 0] = fmaf(kv.x, vj, gv.x * x[4 * i + 0]);
          x[4 * i + 1] = fmaf(kv.y, vj, gv.y * x[4 * i + 1]);
          x[4 * i + 2] = fmaf(kv.z, vj, gv.z * x[4 * i + 2]);
          x[4 * i + 3] = fmaf(kv.w, vj, gv.w * x[4 * i + 3]);
        }
        tprod *= sg[t][jS];
      }
      if (want_o) {
        const float4 *q4 = reinterpret_cast<const float4 *>(sq[t]);
        float o0 = 0.f, o1 = 0.f, o2 = 0.f, o3 = 0.f;
#pragma unroll
        for (int i = 0; i < D / 4; ++i) {
          const float4 qv = q4[i];
          o0 = fmaf(qv.x, x[4 * i + 0], o0);
          o1 = fmaf(qv.y, x[4 * i + 1], o1);
          o2 = fmaf(qv.z, x[4 * i + 2], o2);
          o3 = fmaf(qv.w, x[4 * i + 3], o3);
        }
        a.o_out[((size_t)tok * H + h) * D + jS] = (o0 + o1) + (o2 + o3);
      }
    }
  }

  if (isT) {
#pragma unroll
    for (int i = 0; i < D; ++i) a.T_out[(sidx + i) * D + j] = x[i];
  } else {
#pragma unroll
    for (int i = 0; i < D; ++i) a.S_out[(sidx + i) * D + jS] = x[i];
    if (build && KIND == KIND_SCALAR && cb == 0 && tid == 0) a.T_out[(size_t)s * H + h] = tprod;
    if (build && KIND == KIND_DIAG) a.T_out[((size_t)s * H + h) * D + jS] = tprod;
  }
}

// Dense families (delta, gated delta, KDA) at d = 128: each state column is split over a lane
// pair, so a thread holds 64 rows instead of 128 and four times as many warps fit on an SM.  Lane
// (column c, half hf) owns rows 8 m + 4 hf .. 8 m + 4 hf + 3 (m = 0..15): the two lanes of a pair
// read adjacent 16-byte pieces of each staged k, q or gate vector (one shared-memory wavefront per
// warp), and every column dot product closes with one shuffle between the pair.
template <int KIND, typename Tin>
__global__ void __launch_bounds__(128) recurrent_pair_kernel(RecurrentArgs a) {
  constexpr int D = 128, CPB = 64;  // columns per block
  constexpr int R = 64;             // rows per thread
  const bool build = a.T_out != nullptr;
  const int ncols = build ? 2 * D : D;
  const int ncb = ncols / CPB;
  const int cb = blockIdx.x % ncb;
  const int rest = blockIdx.x / ncb;
  const int h = rest % a.H;
  const int s = rest / a.H;
  const int H = a.H;
  const int tid = threadIdx.x, hf = tid & 1;
  const int j = cb * CPB + (tid >> 1);  // column of the (augmented) state
  const bool isT = build && j < D;      // uniform over the block
  const int jS = build ? j - D : j;

  int64_t beg, end;
  bool ok;
  seg_range(a.seg, s, beg, end, ok);
  if (!ok) {
    if (tid == 0 && cb == 0) set_error(a.err, HYPIC_EDEVICE);
    return;
  }
  const int64_t len = end - beg;

  __shared__ __align__(16) float sk[kTile][D];
  __shared__ __align__(16) float sq[kTile][D];
  __shared__ __align__(16) float sg[kTile][KIND == KIND_KDA ? D : 4];
  __shared__ float sa[kTile], sb[kTile];

  const Tin *K = static_cast<const Tin *>(a.src.k);
  const Tin *V = static_cast<const Tin *>(a.src.v);
  const Tin *Q = static_cast<const Tin *>(a.src.q);
  const bool want_o = (a.o_out != nullptr) && !isT;
  const int fam = a.fam;

  float x[R];  // x[4 m + e] = row 8 m + 4 hf + e
  const size_t sidx = ((size_t)s * H + h) * D;
#pragma unroll
  for (int m = 0; m < 16; ++m)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int i = 8 * m + 4 * hf + e;
      if (isT) x[4 * m + e] = (i == j) ? 1.f : 0.f;
      else x[4 * m + e] = a.S_in ? a.S_in[(sidx + i) * D + jS] : 0.f;
    }

  for (int64_t t0 = 0; t0 < len; t0 += kTile) {
    const int nt = (len - t0 < kTile) ? (int)(len - t0) : kTile;
    __syncthreads();
    for (int e = tid; e < nt * D; e += 128) {
      const int t = e / D, i = e % D;
      const size_t g = ((size_t)(beg + t0 + t) * H + h) * D + i;
      sk[t][i] = to_f32<Tin>(K[g]);
      if (want_o) sq[t][i] = to_f32<Tin>(Q[g]);
      if (KIND == KIND_KDA) sg[t][i] = a.src.alpha[g];
    }
    for (int t = tid; t < nt; t += 128) {
      const size_t g = (size_t)(beg + t0 + t) * H + h;
      sa[t] = fam == HYPIC_FAM_GATED_DELTA ? a.src.alpha[g] : 1.f;
      sb[t] = a.src.beta[g];
    }
    __syncthreads();
    for (int t = 0; t < nt; ++t) {
      const int64_t tok = beg + t0 + t;
      const float vj = isT ? 0.f : to_f32<Tin>(V[((size_t)tok * H + h) * D + jS]);
      const float4 *k4 = reinterpret_cast<const float4 *>(sk[t]) + hf;
      float c0 = 0.f, c1 = 0.f, c2 = 0.f, c3 = 0.f;
      if (KIND == KIND_KDA) {
        const float4 *g4 = reinterpret_cast<const float4 *>(sg[t]) + hf;
#pragma unroll
        for (int m = 0; m < 16; ++m) {
          const float4 kv = k4[2 * m], gv = g4[2 * m];
          x[4 * m + 0] *= gv.x;
          x[4 * m + 1] *= gv.y;
          x[4 * m + 2] *= gv.z;
          x[4 * m + 3] *= gv.w;
          c0 = fmaf(kv.x, x[4 * m + 0], c0);
          c1 = fmaf(kv.y, x[4 * m + 1], c1);
          c2 = fmaf(kv.z, x[4 * m + 2], c2);
          c3 = fmaf(kv.w, x[4 * m + 3], c3);
        }
      } else {
#pragma unroll
        for (int m = 0; m < 16; ++m) {
          const float4 kv = k4[2 * m];
          c0 = fmaf(kv.x, x[4 * m + 0], c0);
          c1 = fmaf(kv.y, x[4 * m + 1], c1);
          c2 = fmaf(kv.z, x[4 * m + 2], c2);
          c3 = fmaf(kv.w, x[4 * m + 3], c3);
        }
      }
      float c = (c0 + c1) + (c2 + c3);
      c += __shfl_xor_sync(0xffffffffu, c, 1);
      // k is read again below rather than held from the loop above: 64 more live registers would
      // cost a quarter of the warps an SM can hold.
      asm volatile("" ::: "memory");
      if (KIND == KIND_KDA) {
        const float coef = sb[t] * (vj - c);
#pragma unroll
        for (int m = 0; m < 16; ++m) {
          const float4 kv = k4[2 * m];
          x[4 * m + 0] = fmaf(coef, kv.x, x[4 * m + 0]);
          x[4 * m + 1] = fmaf(coef, kv.y, x[4 * m + 1]);
          x[4 * m + 2] = fmaf(coef, kv.z, x[4 * m + 2]);
          x[4 * m + 3] = fmaf(coef, kv.w, x[4 * m + 3]);
        }
      } else {
        const float at = sa[t];
        const float coef = sb[t] * (vj - at * c);
#pragma unroll
        for (int m = 0; m < 16; ++m) {
          const float4 kv = k4[2 * m];
          x[4 * m + 0] = fmaf(coef, kv.x, at * x[4 * m + 0]);
          x[4 * m + 1] = fmaf(coef, kv.y, at * x[4 * m + 1]);
          x[4 * m + 2] = fmaf(coef, kv.z, at * x[4 * m + 2]);
          x[4 * m + 3] = fmaf(coef, kv.w, at * x[4 * m + 3]);
        }
      }
      if (want_o) {
        const float4 *q4 = reinterpret_cast<const float4 *>(sq[t]) + hf;
        float o0 = 0.f, o1 = 0.f, o2 = 0.f, o3 = 0.f;
#pragma unroll
        for (int m = 0; m < 16; ++m) {
          const float4 qv = q4[2 * m];
          o0 = fmaf(qv.x, x[4 * m + 0], o0);
          o1 = fmaf(qv.y, x[4 * m + 1], o1);
          o2 = fmaf(qv.z, x[4 * m + 2], o2);
          o3 = fmaf(qv.w, x[4 * m + 3], o3);
        }
        float o = (o0 + o1) + (o2 + o3);
        o += __shfl_xor_sync(0xffffffffu, o, 1);
        if (hf == 0) a.o_out[((size_t)tok * H + h) * D + jS] = o;
      }
    }
  }

  float *out = isT ? a.T_out + (sidx) * D + j : a.S_out + (sidx) * D + jS;
#pragma unroll
  for (int m = 0; m < 16; ++m)
#pragma unroll
    for (int e = 0; e < 4; ++e) out[(size_t)(8 * m + 4 * hf + e) * D] = x[4 * m + e];
}

template <int D, typename Tin>
cudaError_t launch_d(const RecurrentArgs &a, cudaStream_t st) {
  constexpr int TPC = D >= 64 ? 64 : D;
  const bool dense = a.fam == HYPIC_FAM_DELTA || a.fam == HYPIC_FAM_GATED_DELTA || a.fam == HYPIC_FAM_KDA;
  const int ncols = (a.T_out && dense) ? 2 * D : D;
  const long long blocks = (long long)a.n_seg * a.H * (ncols / TPC);
  if (blocks <= 0) return cudaSuccess;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  if (D == 128 && dense) {
    // lane-pair kernel: 64 columns per 128-thread block, the same block count
    if (a.fam == HYPIC_FAM_KDA)
      recurrent_pair_kernel<KIND_KDA, Tin><<<(unsigned)blocks, 128, 0, st>>>(a);
    else
      recurrent_pair_kernel<KIND_DELTA, Tin><<<(unsigned)blocks, 128, 0, st>>>(a);
    return cudaGetLastError();
  }
  if (a.fam == HYPIC_FAM_KDA)
    recurrent_kernel<D, KIND_KDA, Tin><<<(unsigned)blocks, TPC, 0, st>>>(a);
  else if (dense)
    recurrent_kernel<D, KIND_DELTA, Tin><<<(unsigned)blocks, TPC, 0, st>>>(a);
  else if (a.fam == HYPIC_FAM_DIAG)
    recurrent_kernel<D, KIND_DIAG, Tin><<<(unsigned)blocks, TPC, 0, st>>>(a);
  else
    recurrent_kernel<D, KIND_SCALAR, Tin><<<(unsigned)blocks, TPC, 0, st>>>(a);
  return cudaGetLastError();
}

template <typename Tin>
cudaError_t launch_t(const RecurrentArgs &a, cudaStream_t st) {
  switch (a.D) {
    case 16: return launch_d<16, Tin>(a, st);
    case 32: return launch_d<32, Tin>(a, st);
    case 64: return launch_d<64, Tin>(a, st);
    case 128: return launch_d<128, Tin>(a, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_recurrent(const RecurrentArgs &a, cudaStream_t st) {
  if (a.src.in_dtype == HYPIC_BF16) return launch_t<__nv_bfloat16>(a, st);
  return launch_t<float>(a, st);
}

}  // namespace hypic
