// Chunked tensor-core segment build for the KDA family at d_k = d_v = 128, bf16 inputs.
//
// What it computes (HYPIC reading notes: Method 2 segment pair; Method 3, Table 1, KDA row):
// (T_C, S_{C|0}) of a segment body for T_i = (I - b_i k_i k_i^T) diag(g_i), u_i = b_i k_i v_i^T,
// as the end value of the augmented state X = [T | S] (d_k x 2d) run from [I | 0].
//
// Chunked form, 64 tokens per chunk.  With G_t = sum_{r<=t} log2 g_r (per key channel, inside the
// chunk), Gamma_t = 2^{G_t}, and the effective writes w_t^T = b_t (v_t^T - k_t^T diag(g_t) S_{t-1}),
// the per-token rule S_t = diag(g_t) S_{t-1} + k_t w_t^T unrolls to
//   (I + L) W = diag(b) V - diag(b) (K o Gamma) X,   L_ts = b_t sum_i k_ti k_si 2^{G_ti - G_si}  (s < t)
//   X_new     = diag(Gamma_C) X + Khat^T (W),          Khat_si = k_si 2^{G_Ci - G_si},
// so with A = (I + L)^{-1}: W = U - Wk X, U = A diag(b) V, Wk = A diag(b) (K o Gamma).
// Against the gated-delta build the decay is per channel: it sits inside the Gram (a product of
// the decayed keys (K o E)(K o F)^T with E_t = 2^{G_t - G_m}, F_s = 2^{G_m - G_s} around the middle
// token m), inside Wk and inside the update's key operand Khat, none of which is exact in bf16, so
// each of those products takes hi and lo pieces; the state's rows are scaled by the vector Gamma_C.
//
// Two kernels per block of heads:
//   kda_prep_kernel  (one CTA per chunk and head, three per SM): the gates' per-channel running
//     products in registers, then the key channels in two halves of 64 (one key box and one E half
//     in shared memory at a time): the decayed Gram on tcgen05 (M = 64, three split products,
//     accumulated over the halves), L, A = (I + L)^{-1} in fp32 (the same blocked inverse as the
//     gated-delta build), Wk^T = (K o Gamma)^T (A diag(b))^T on tcgen05, and Khat.  Stored as a
//     record of ready-made 128-byte-swizzled operand tiles: Wk^T hi + lo, -A diag(b) hi + lo,
//     Khat hi + lo, and Gamma_C.
//   chain_kda_kernel (one CTA per segment, head and column half): the state-dependent chain with
//     that half's X^T (and its hi and lo pieces) in tensor memory: per chunk P^T = X^T Wk^T (minus
//     U^T = V^T (A diag(b))^T for the S half), X^T <- X^T diag(Gamma_C) + R^T Khat with
//     R^T = -(P^T - U^T) in hi + lo pieces.  The record is too large for both halves and two stages
//     in one CTA's shared memory, so each half runs in its own CTA.
// Padded tokens of a ragged last chunk get b = 0 and g = 1, which makes them exact identity steps.
// A chunk whose per-channel decay spans 2^100 or more in some channel (far stronger gates than any
// workload here) forms L on the CUDA cores with one exponential per term instead of the factored
// Gram, so no factor leaves the fp32 range.
#include <cuda_bf16.h>

#include "tc_ptx.cuh"
#include "tma_host.h"

namespace hypic {
namespace {

using namespace tc;

constexpr int C = 64;    // tokens per chunk
constexpr int D = 128;   // d_k = d_v
constexpr int NT = 128;  // prep threads

// Record of one (chunk, head), byte offsets.  Wk^T: MN-major [128 i][64 t] tiles; -A diag(b):
// K-major [64 t][64 s] tiles; Khat: two [64 t][64 i] boxes per piece (the K tile's layout);
// Gamma_C: 128 floats.
constexpr uint32_t KR_WH = 0, KR_WL = 16384, KR_AVH = 32768, KR_AVL = 40960, KR_KH = 49152, KR_KL = 65536;
constexpr uint32_t KR_GC = 81920;
constexpr uint32_t KR_REC = KR_GC + 512;  // 82,432 bytes
constexpr size_t KWS_CAP = (size_t)4 << 30;  // preferred workspace size bound

struct KdaArgs {
  int H;       // heads of the token tensors
  int h0, Hb;  // this launch covers heads [h0, h0 + Hb)
  int n_seg;
  const int64_t *bounds;  // [n_seg][2] or null: single segment [0, len0)
  int64_t len0, max_len, n_tokens;
  int max_chunks;
  const float *alpha;  // channel gates [tokens, H, D]
  const float *beta;   // [tokens, H]
  float *T_out, *S_out;
  uint8_t *ws;
  int *err;
};

__device__ __forceinline__ bool kseg_bounds(const KdaArgs &a, int s, int64_t &beg, int64_t &end) {
  if (a.bounds) {
    beg = a.bounds[2 * s];
    end = a.bounds[2 * s + 1];
  } else {
    beg = 0;
    end = a.len0;
  }
  return beg >= 0 && end >= beg && end - beg <= a.max_len && end <= a.n_tokens;
}

__device__ __forceinline__ uint8_t *krec(const KdaArgs &a, int s, int c, int hh) {
  return a.ws + (((size_t)s * a.max_chunks + c) * a.Hb + hh) * KR_REC;
}

// Byte offset of element (t, i) in a [64 t][128 i] bf16 tile stored as two 128-byte-swizzled
// [64 t][64 i] boxes (the layout the TMA writes the key chunk in).
__device__ __forceinline__ uint32_t kt_off(int t, int i) {
  return (uint32_t)(i >> 6) * 8192u + sw128_offset((uint32_t)t, (uint32_t)((i & 63) >> 3)) + (uint32_t)(i & 7) * 2u;
}
__device__ __forceinline__ float kt_get(const uint8_t *tile, int t, int i) {
  return __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(tile + kt_off(t, i)));
}

// hi = bf16(v), lo = bf16(v - hi) for 8 values, packed for one 16-byte store each.
__device__ __forceinline__ void ksplit8(const float *v, uint4 &hi, uint4 &lo) {
  uint32_t h[4], l[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const __nv_bfloat162 hp = __floats2bfloat162_rn(v[2 * q], v[2 * q + 1]);
    const float2 hf = __bfloat1622float2(hp);
    const __nv_bfloat162 lp = __floats2bfloat162_rn(v[2 * q] - hf.x, v[2 * q + 1] - hf.y);
    h[q] = *reinterpret_cast<const uint32_t *>(&hp);
    l[q] = *reinterpret_cast<const uint32_t *>(&lp);
  }
  hi = make_uint4(h[0], h[1], h[2], h[3]);
  lo = make_uint4(l[0], l[1], l[2], l[3]);
}

// hi = truncation of x to bf16, lo = bf16 rounding of the exact remainder, for two values.
__device__ __forceinline__ void ksplit2(float a, float b, uint32_t &hi, uint32_t &lo) {
  const uint32_t ua = __float_as_uint(a), ub = __float_as_uint(b);
  const float ra = a - __uint_as_float(ua & 0xFFFF0000u), rb = b - __uint_as_float(ub & 0xFFFF0000u);
  hi = __byte_perm(ua, ub, 0x7632);
  const __nv_bfloat162 lp = __floats2bfloat162_rn(ra, rb);
  lo = *reinterpret_cast<const uint32_t *>(&lp);
}

// ------------------------------------------------------------------------------------------------
// Kernel 1: per (segment, chunk, head).  Shared memory is held to 72 KB, three CTAs per SM: the
// gates are read straight into registers (thread = key channel), and the key channels are worked
// through in two halves of 64, each with its key box and its E (or G) half in shared memory; the
// Gram accumulates over the halves, (K o E) is kept whole for Wk^T, (K o F) one half at a time.
constexpr int LS = 68;  // row stride of L (floats)
constexpr uint32_t KP_KB = 0;        // key box of the current channel half, [64 t][64 i] bf16 (TMA)
constexpr uint32_t KP_EH = 8192;     // E (or G) of the current channel half, fp32 [64 t][64 i];
                                     // after both halves L, A, then A diag(b) hi and lo (from KP_KB)
constexpr uint32_t KP_P1H = 24576;   // (K o E) hi, lo: two boxes each; the Gram's first operand and
constexpr uint32_t KP_P1L = 40960;   // Wk^T's; then Wk^T hi, lo staged for the store
constexpr uint32_t KP_P2H = 57344;   // (K o F) hi, lo of the current half: the Gram's second operand;
constexpr uint32_t KP_P2L = 65536;   // fallback: L (s < t) accumulated over the halves, row stride 64
constexpr uint32_t KP_SMEM = 73728;  // 1024-aligned base (declared alignment), no slack

__global__ void __launch_bounds__(NT, 3)
    kda_prep_kernel(const __grid_constant__ CUtensorMap mapK, const __grid_constant__ KdaArgs a) {
  extern __shared__ __align__(1024) uint8_t sm[];
  __shared__ uint64_t bar_tma, bar_mma;
  __shared__ uint32_t tmem_slot;
  __shared__ float sBv[C];
  __shared__ int ok_flag;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int hh = blockIdx.x % a.Hb;
  const int c = (blockIdx.x / a.Hb) % a.max_chunks;
  const int s = (blockIdx.x / a.Hb) / a.max_chunks;
  const int h = a.h0 + hh;
  int64_t beg, end;
  if (!kseg_bounds(a, s, beg, end)) return;  // reported by the chain kernel
  if ((int64_t)c * C >= end - beg) return;
  if ((smem_u32(sm) & 1023u) != 0) {  // the swizzled tiles need a 1024-byte aligned base
    if (tid == 0) set_error(a.err, HYPIC_EDEVICE);
    return;
  }
  const int64_t t0 = beg + (int64_t)c * C;
  const int nvalid = (int)((end - t0) < C ? (end - t0) : C);

  if (tid == 0) {
    mbar_init(&bar_tma, 1);
    mbar_init(&bar_mma, 1);
    mbar_fence_init();
    ok_flag = 1;
    mbar_arrive_expect_tx(&bar_tma, 8192);
    tma_load_2d(sm + KP_KB, &mapK, &bar_tma, h * D, (int)t0);
  }
  if (warp == 0) {
    tmem_alloc(&tmem_slot, 64);
    tmem_relinquish();
  }
  if (tid < C) sBv[tid] = tid < nvalid ? a.beta[(t0 + tid) * a.H + h] : 0.f;

  // Thread = key channel i: Gamma_t = running product of the channel's gates (tokens past the body
  // count as gate 1), in registers, the gates read row by row (each row coalesced over the
  // channels).  Gamma_0 / Gamma_{C-1} <= 1 / Gamma_{C-1}: factors around the middle stay within
  // 2^100 when Gamma_{C-1} >= 2^-100 in every channel (separable).  Then E_t = Gamma_t / M with
  // M = 2^round(log2 Gamma_m) at the middle token, a power of two, so E_t and the rescaling of
  // Wk^T's rows by M are exact.  Otherwise (the fallback) G_t, the log2-cumsum of the gates, and
  // every factor is one exponential.
  const int ch = tid;
  const float *gp = a.alpha + ((size_t)t0 * a.H + h) * D + ch;
  const size_t gstride = (size_t)a.H * D;
  float gv[C];
#pragma unroll
  for (int t = 0; t < C; ++t) gv[t] = t < nvalid ? __ldg(gp + (size_t)t * gstride) : 1.f;
  float GamC;
  {
    float pr = 1.f;
#pragma unroll
    for (int t = 0; t < C; ++t) {
      pr *= gv[t];
      gv[t] = pr;
    }
    GamC = pr;
  }
  const bool separable = __syncthreads_and(GamC >= 0x1p-100f) != 0;
  float wk_scale = 1.f;
  if (separable) {
    const int em = (int)rintf(log2f(gv[C / 2]));
    const float Minv = ldexpf(1.f, -em);
    wk_scale = ldexpf(1.f, em);
#pragma unroll
    for (int t = 0; t < C; ++t) gv[t] *= Minv;
  } else {
    float g = 0.f;
#pragma unroll
    for (int t = 0; t < C; ++t) {
      g += t < nvalid ? log2f(__ldg(gp + (size_t)t * gstride)) : 0.f;
      gv[t] = g;
    }
  }
  uint8_t *rec = krec(a, s, c, hh);
  reinterpret_cast<float *>(rec + KR_GC)[ch] = GamC;
  tc_fence_after();
  const uint32_t tmem = tmem_slot;  // written before the barrier above
  const uint8_t *sK = sm + KP_KB;
  float *sE = reinterpret_cast<float *>(sm + KP_EH);  // [64 t][64 i], the current half
  float *sLacc = reinterpret_cast<float *>(sm + KP_P2H);  // fallback: [64 t][64 s]

  // The two channel halves.  Per half: E (or G) to shared memory, then one pass over the half's
  // 64 x 64 entries, eight channels of one token per item: the Gram's operands (K o E) (also
  // Wk^T's, rescaled by M per channel afterwards) and (K o F), F = 1 / E, in hi and lo pieces, and
  // Khat = K o Gamma_C / Gamma = (K o F) E_{C-1} straight to the record (the quotient by the fast
  // reciprocal: its error, about 2^-22, is far below the hi + lo split's); then the half's Gram
  // products.  Fallback: (K o E) = K o 2^G, Khat = K o 2^{G_{C-1} - G}, and the half's share of
  // L_ts = b_t sum_i k_ti k_si 2^{G_ti - G_si} term by term.
#pragma unroll 1
  for (int hf = 0; hf < 2; ++hf) {
    if ((ch >> 6) == hf) {
#pragma unroll
      for (int t = 0; t < C; ++t) sE[t * 64 + (ch & 63)] = gv[t];
    }
    __syncthreads();
    // every thread reads the key box (and, before the second half's pass overwrites (K o F), the
    // first half's Gram products must have read it)
    bool got = mbar_wait_cycles(&bar_tma, (uint32_t)hf, tid == 0 ? a.err : nullptr);
    if (separable && hf == 1) got = got && mbar_wait_cycles(&bar_mma, 0u, tid == 0 ? a.err : nullptr);
    if (!got) ok_flag = 0;
    __syncthreads();
    if (!ok_flag) break;
    const int c8 = tid & 7;  // channel octet within the half
    float L8[8];
    {
      const float4 e0 = *reinterpret_cast<const float4 *>(sE + (C - 1) * 64 + 8 * c8);
      const float4 e1 = *reinterpret_cast<const float4 *>(sE + (C - 1) * 64 + 8 * c8 + 4);
      L8[0] = e0.x; L8[1] = e0.y; L8[2] = e0.z; L8[3] = e0.w;
      L8[4] = e1.x; L8[5] = e1.y; L8[6] = e1.z; L8[7] = e1.w;
    }
#pragma unroll 2
    for (int j = 0; j < 4; ++j) {
      const int t = (tid >> 3) + 16 * j;  // token of item tid + 128 j
      const uint32_t off = sw128_offset((uint32_t)t, (uint32_t)c8);
      const uint4 kr = *reinterpret_cast<const uint4 *>(sK + off);
      const __nv_bfloat162 *k2 = reinterpret_cast<const __nv_bfloat162 *>(&kr);
      const float4 g0 = *reinterpret_cast<const float4 *>(sE + t * 64 + 8 * c8);
      const float4 g1 = *reinterpret_cast<const float4 *>(sE + t * 64 + 8 * c8 + 4);
      const float G8[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
      float k8[8], p1[8], p2[8], kh[8];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float2 kv = __bfloat1622float2(k2[q]);
        k8[2 * q] = kv.x;
        k8[2 * q + 1] = kv.y;
      }
      if (separable) {
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          p1[q] = k8[q] * G8[q];
          p2[q] = __fdividef(k8[q], G8[q]);
          kh[q] = p2[q] * L8[q];
        }
      } else {
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          p1[q] = k8[q] * exp2f(G8[q]);
          p2[q] = 0.f;
          kh[q] = k8[q] * exp2f(L8[q] - G8[q]);
        }
      }
      const uint32_t boff = (uint32_t)hf * 8192u + off;
      uint4 hi, lo;
      ksplit8(p1, hi, lo);
      *reinterpret_cast<uint4 *>(sm + KP_P1H + boff) = hi;
      *reinterpret_cast<uint4 *>(sm + KP_P1L + boff) = lo;
      if (separable) {
        ksplit8(p2, hi, lo);
        *reinterpret_cast<uint4 *>(sm + KP_P2H + off) = hi;
        *reinterpret_cast<uint4 *>(sm + KP_P2L + off) = lo;
      }
      ksplit8(kh, hi, lo);
      *reinterpret_cast<uint4 *>(rec + KR_KH + boff) = hi;
      *reinterpret_cast<uint4 *>(rec + KR_KL + boff) = lo;
    }
    if (!separable) {
      // thread pair (t, half of the half's channels), adjacent lanes: sum over 32 channels each,
      // the pair reduced by a shuffle; only the strict lower triangle is kept (the inverse reads
      // nothing else)
      const int t = tid >> 1, ih = tid & 1;
      for (int s2 = 0; s2 < C; ++s2) {
        float acc = 0.f;
        if (s2 < t) {
          for (int i = 32 * ih; i < 32 * ih + 32; ++i) {
            const float kk = kt_get(sK, t, i) * kt_get(sK, s2, i);
            acc = fmaf(kk, exp2f(sE[t * 64 + i] - sE[s2 * 64 + i]), acc);
          }
        }
        acc += __shfl_xor_sync(0xffffffffu, acc, 1);
        if (ih == 0 && s2 < t) sLacc[t * 64 + s2] = hf ? sLacc[t * 64 + s2] + acc : acc;
      }
    }
    fence_proxy_async();
    __syncthreads();  // the half's operands are written; its key box and E are read
    if (tid == 0) {
      tc_fence_after();
      if (separable) {
        // Gram += (K o E)(K o F)^T over the half's channels (M = 64, N = 64, K = 64); three products
        const uint32_t id = idesc_f32acc(1, 1, 0, 0, 64, 64);
        const uint32_t p1h = smem_u32(sm + KP_P1H) + hf * 8192, p1l = smem_u32(sm + KP_P1L) + hf * 8192;
        const uint32_t p2h = smem_u32(sm + KP_P2H), p2l = smem_u32(sm + KP_P2L);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint32_t o = kk * 32;
          const uint64_t ah = sdesc_sw128(p1h + o, 16, 1024), al = sdesc_sw128(p1l + o, 16, 1024);
          const uint64_t bh = sdesc_sw128(p2h + o, 16, 1024), bl = sdesc_sw128(p2l + o, 16, 1024);
          mma_f16(tmem, ah, bh, id, (hf | kk) != 0);
          mma_f16(tmem, ah, bl, id, 1);
          mma_f16(tmem, al, bh, id, 1);
        }
        mma_commit(&bar_mma);
      }
      if (hf == 0) {
        // the second key box, into the first one's buffer (all of its reads are done)
        mbar_arrive_expect_tx(&bar_tma, 8192);
        tma_load_2d(sm + KP_KB, &mapK, &bar_tma, h * D + 64, (int)t0);
      }
    }
  }
  if (separable && tid == 0 && ok_flag && !mbar_wait_cycles(&bar_mma, 1u, a.err)) ok_flag = 0;
  __syncthreads();  // the Gram (or the fallback's L) is complete
  tc_fence_after();

  float *sL = reinterpret_cast<float *>(sm + KP_KB);  // over the key box and E, both read
  float *sA = sL;
  float *sT = sL + 32;
  if (ok_flag) {
    if (separable) {
      // L_ts = b_t Gram_ts (s < t).  Gram row t sits in lane 32 (t / 16) + t % 16 (16x256b load).
      const int ta = warp * 16 + (lane >> 2), tb = ta + 8, cq = 2 * (lane & 3);
      float v[32];
      tmem_ld16x256_x8(tmem + ((uint32_t)(warp * 32) << 16), v);
      const float ba = sBv[ta], bb = sBv[tb];
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        const int sc = 8 * m + cq;
        *reinterpret_cast<float2 *>(sL + ta * LS + sc) =
            make_float2(sc < ta ? ba * v[4 * m] : 0.f, sc + 1 < ta ? ba * v[4 * m + 1] : 0.f);
        *reinterpret_cast<float2 *>(sL + tb * LS + sc) =
            make_float2(sc < tb ? bb * v[4 * m + 2] : 0.f, sc + 1 < tb ? bb * v[4 * m + 3] : 0.f);
      }
    } else {
      // L_ts = b_t (sum over both halves), s < t, from the accumulated rows
      for (int e = tid; e < C * C; e += NT) {
        const int t = e >> 6, s2 = e & 63;
        if (s2 < t) sL[t * LS + s2] = sBv[t] * sLacc[t * 64 + s2];
      }
    }
  }
  __syncthreads();
  if (!ok_flag) {
    if (warp == 0) tmem_dealloc(tmem, 64);
    return;
  }

  // A = (I + L)^{-1}, unit lower triangular, in place over L (rows stride LS): 16 x 16 diagonal
  // blocks by forward substitution, then the 32 x 32 and 64 x 64 levels by block products.
  {
    float x[16];
    const int base = (tid >> 4) * 16, cl = tid & 15;
    if (tid < C) {
#pragma unroll
      for (int r = 0; r < 16; ++r) x[r] = (r == cl) ? 1.f : 0.f;
#pragma unroll
      for (int r = 1; r < 16; ++r) {
        const float *Lr = sL + (base + r) * LS + base;
        float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
        for (int q = 0; q + 3 < r; q += 4) {
          const float4 l4 = *reinterpret_cast<const float4 *>(Lr + q);
          a0 = fmaf(l4.x, x[q], a0);
          a1 = fmaf(l4.y, x[q + 1], a1);
          a2 = fmaf(l4.z, x[q + 2], a2);
          a3 = fmaf(l4.w, x[q + 3], a3);
        }
#pragma unroll
        for (int q = (r / 4) * 4; q < r; ++q) a0 = fmaf(Lr[q], x[q], a0);
        if (r > cl) x[r] = -((a0 + a1) + (a2 + a3));
      }
    }
    __syncthreads();
    if (tid < C) {
#pragma unroll
      for (int r = 0; r < 16; ++r) sA[(base + r) * LS + base + cl] = x[r];
    }
  }
  __syncthreads();
  {
    const int p = tid >> 6, r = (tid & 63) >> 2, c0 = 4 * (tid & 3);
    const int o = 32 * p;
    float4 y = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const float l = sL[(o + 16 + r) * LS + o + k];
      const float4 a4 = *reinterpret_cast<const float4 *>(sA + (o + k) * LS + o + c0);
      y.x = fmaf(l, a4.x, y.x);
      y.y = fmaf(l, a4.y, y.y);
      y.z = fmaf(l, a4.z, y.z);
      y.w = fmaf(l, a4.w, y.w);
    }
    float *Y = sT + 16 * p;
    *reinterpret_cast<float4 *>(Y + r * LS + c0) = y;
    __syncthreads();
    float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const float ab = sA[(o + 16 + r) * LS + o + 16 + k];
      const float4 y4 = *reinterpret_cast<const float4 *>(Y + k * LS + c0);
      z.x = fmaf(ab, y4.x, z.x);
      z.y = fmaf(ab, y4.y, z.y);
      z.z = fmaf(ab, y4.z, z.z);
      z.w = fmaf(ab, y4.w, z.w);
    }
    *reinterpret_cast<float4 *>(sA + (o + 16 + r) * LS + o + c0) = make_float4(-z.x, -z.y, -z.z, -z.w);
  }
  __syncthreads();
  {
    const int r0 = 2 * (tid >> 3), c0 = 4 * (tid & 7);
    float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll 8
    for (int k = 0; k < 32; ++k) {
      const float a0 = sL[(32 + r0) * LS + k], a1 = sL[(33 + r0) * LS + k];
      const float4 b4 = *reinterpret_cast<const float4 *>(sA + k * LS + c0);
      acc[0][0] = fmaf(a0, b4.x, acc[0][0]);
      acc[0][1] = fmaf(a0, b4.y, acc[0][1]);
      acc[0][2] = fmaf(a0, b4.z, acc[0][2]);
      acc[0][3] = fmaf(a0, b4.w, acc[0][3]);
      acc[1][0] = fmaf(a1, b4.x, acc[1][0]);
      acc[1][1] = fmaf(a1, b4.y, acc[1][1]);
      acc[1][2] = fmaf(a1, b4.z, acc[1][2]);
      acc[1][3] = fmaf(a1, b4.w, acc[1][3]);
    }
    *reinterpret_cast<float4 *>(sT + r0 * LS + c0) = make_float4(acc[0][0], acc[0][1], acc[0][2], acc[0][3]);
    *reinterpret_cast<float4 *>(sT + (r0 + 1) * LS + c0) = make_float4(acc[1][0], acc[1][1], acc[1][2], acc[1][3]);
    __syncthreads();
    float bcc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    const int kmax = 8 * warp + 8;
#pragma unroll 8
    for (int k = 0; k < kmax; ++k) {
      const float a0 = sA[(32 + r0) * LS + 32 + k], a1 = sA[(33 + r0) * LS + 32 + k];
      const float4 b4 = *reinterpret_cast<const float4 *>(sT + k * LS + c0);
      bcc[0][0] = fmaf(a0, b4.x, bcc[0][0]);
      bcc[0][1] = fmaf(a0, b4.y, bcc[0][1]);
      bcc[0][2] = fmaf(a0, b4.z, bcc[0][2]);
      bcc[0][3] = fmaf(a0, b4.w, bcc[0][3]);
      bcc[1][0] = fmaf(a1, b4.x, bcc[1][0]);
      bcc[1][1] = fmaf(a1, b4.y, bcc[1][1]);
      bcc[1][2] = fmaf(a1, b4.z, bcc[1][2]);
      bcc[1][3] = fmaf(a1, b4.w, bcc[1][3]);
    }
    *reinterpret_cast<float4 *>(sA + (32 + r0) * LS + c0) = make_float4(-bcc[0][0], -bcc[0][1], -bcc[0][2], -bcc[0][3]);
    *reinterpret_cast<float4 *>(sA + (33 + r0) * LS + c0) = make_float4(-bcc[1][0], -bcc[1][1], -bcc[1][2], -bcc[1][3]);
  }
  __syncthreads();

  // A diag(b) split hi + lo: K-major [64 t][64 s] tiles, to shared memory (over A, once all of A
  // is read) for the Wk^T product, and negated to the record for the chain's U product.
  uint8_t *ab_tiles = reinterpret_cast<uint8_t *>(sL);  // 1024-aligned: KP_KB
  uint4 abh[4], abl[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int e = tid + j * NT;
    const int t = e >> 3, q = e & 7;
    float vb[8], vv[8];
    const float4 a0 = *reinterpret_cast<const float4 *>(sA + t * LS + 8 * q);
    const float4 a1 = *reinterpret_cast<const float4 *>(sA + t * LS + 8 * q + 4);
    const float av8[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float av = (8 * q + i <= t) ? av8[i] : 0.f;
      vb[i] = av * sBv[8 * q + i];
      vv[i] = -vb[i];
    }
    uint4 hi, lo;
    const uint32_t off = sw128_offset((uint32_t)t, (uint32_t)q);
    ksplit8(vb, abh[j], abl[j]);
    ksplit8(vv, hi, lo);
    *reinterpret_cast<uint4 *>(rec + KR_AVH + off) = hi;
    *reinterpret_cast<uint4 *>(rec + KR_AVL + off) = lo;
  }
  __syncthreads();
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int e = tid + j * NT;
    const uint32_t off = sw128_offset((uint32_t)(e >> 3), (uint32_t)(e & 7));
    *reinterpret_cast<uint4 *>(ab_tiles + off) = abh[j];
    *reinterpret_cast<uint4 *>(ab_tiles + 8192 + off) = abl[j];
  }
  fence_proxy_async();
  __syncthreads();

  if (tid == 0) {
    // Wk^T' = (K o E)^T (A diag(b))^T: M = 128 (i), N = 64 (t), K = 64 (s); three split products.
    // Row i times 2^{G_m,i} (exact) is Wk^T = (K o Gamma)^T (A diag(b))^T.
    tc_fence_after();
    const uint32_t kh = smem_u32(sm + KP_P1H), kl = smem_u32(sm + KP_P1L), ab = smem_u32(ab_tiles);
    const uint32_t id = idesc_f32acc(1, 1, 1, 0, 128, 64);  // A MN-major, B K-major
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      const uint64_t akh = sdesc_sw128(kh + kk * 2048, 8192, 1024);
      const uint64_t akl = sdesc_sw128(kl + kk * 2048, 8192, 1024);
      const uint64_t bh = sdesc_sw128(ab + kk * 32, 16, 1024);
      const uint64_t bl = sdesc_sw128(ab + 8192 + kk * 32, 16, 1024);
      mma_f16(tmem, akh, bh, id, kk > 0);
      mma_f16(tmem, akh, bl, id, 1);
      mma_f16(tmem, akl, bh, id, 1);
    }
    mma_commit(&bar_mma);
    // the Gram, when formed on the tensor cores, took the barrier's first two phases: this is
    // phase 2 then (or 0), parity 0 either way
    if (!mbar_wait_cycles(&bar_mma, 0u, a.err)) ok_flag = 0;
  }
  __syncthreads();
  tc_fence_after();
  if (ok_flag) {
    // lane i = tid holds row i: MN-major [128 i][64 t] hi and lo tiles over (K o E).
    const float sc = wk_scale;
#pragma unroll 1
    for (int hb = 0; hb < C; hb += 32) {
      float wv[32];
      tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + hb, wv);
#pragma unroll
      for (int q = 0; q < 32; ++q) wv[q] *= sc;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint4 hi, lo;
        ksplit8(wv + 8 * q, hi, lo);
        const uint32_t off = sw128_offset((uint32_t)tid, (uint32_t)(hb / 8 + q));
        *reinterpret_cast<uint4 *>(sm + KP_P1H + off) = hi;
        *reinterpret_cast<uint4 *>(sm + KP_P1L + off) = lo;
      }
    }
  }
  fence_proxy_async();
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 64);
  if (tid == 0 && ok_flag) {
    bulk_store(rec + KR_WH, sm + KP_P1H, 32768);
    bulk_store_commit();
    bulk_store_wait_read();  // the shared source must outlive the copy
  }
}

// ------------------------------------------------------------------------------------------------
// Kernel 2: per (segment, head, column half) -- the chunk chain on tensor memory.
//
// The half's state is kept transposed, X^T (lanes = its 128 columns n, TMEM columns = rows i):
//   P^T - U^T = X^T Wk^T - U^T     A = X^T hi / lo pieces (TMEM), B = Wk^T [i][t] (MN-major)
//   X^T = X^T diag(Gamma_C) + R^T Khat,  R^T = -(P^T - U^T) in hi / lo pieces (TMEM, over P^T)
// -U^T = V^T (-A diag(b))^T goes into the S half's P accumulator first.  Warp 8 issues the MMAs,
// warp 9 the copies, warps 0-7 convert (two threads per TMEM lane, each half the columns).
constexpr uint32_t ST_V = 81920;   // V chunk, two [64 t][64 j] boxes (S half)
constexpr uint32_t ST_GC = 98304;  // Gamma_C, 128 floats
constexpr uint32_t ST_BYTES = 99328;
constexpr uint32_t KC_SMEM = 2 * ST_BYTES + 1024;
constexpr uint32_t TX = 0, TXH = 128, TXL = 192, TP = 256;  // TMEM columns
constexpr int KNC = 256;         // conversion threads
constexpr int KNT = KNC + 64;    // + MMA warp + copy warp

__global__ void __launch_bounds__(KNT, 1)
    chain_kda_kernel(const __grid_constant__ CUtensorMap mapV, const __grid_constant__ KdaArgs a) {
  extern __shared__ uint8_t smem_raw[];
  // r1[b]: the state pieces of column block b written (block 0: each thread's first 32 columns)
  __shared__ uint64_t bar_full[2], bar_empty[2], bar_r1[2], bar_r2, bar_p, bar_x;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(sm);
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int half = blockIdx.x & 1;  // 0: T columns, 1: S columns
  const int unit = blockIdx.x >> 1;
  const int hh = unit % a.Hb, s = unit / a.Hb, h = a.h0 + hh;
  int64_t beg, end;
  if (!kseg_bounds(a, s, beg, end)) {
    if (tid == 0) set_error(a.err, HYPIC_EDEVICE);
    return;
  }
  const int nch = (int)((end - beg + C - 1) / C);
  float *out = (half ? a.S_out : a.T_out) + ((size_t)s * a.H + h) * D * D;
  const int row = tid & 127, part = (tid >> 7) & 1;
  if (nch == 0) {
    // empty body: the identity pair
    if (tid < KNC)
      for (int i = 64 * part; i < 64 * part + 64; ++i) out[(size_t)i * D + row] = (half == 0 && i == row) ? 1.f : 0.f;
    return;
  }

  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar_full[i], 1);
      mbar_init(&bar_empty[i], 1);
    }
    mbar_init(&bar_r1[0], KNC);
    mbar_init(&bar_r1[1], KNC);
    mbar_init(&bar_r2, KNC);
    mbar_init(&bar_p, 1);
    mbar_init(&bar_x, 1);
    mbar_fence_init();
    abort_flag = 0;
  }
  if (warp == 0) {
    tmem_alloc(&tmem_slot, 512);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;

  if (warp == 9) {
    // ---------------------------------------------------------------------------- copy warp
    if (lane == 0) {
      if (half) prefetch_tmap(&mapV);
      const uint32_t bytes = half ? KR_GC + 16384u + 512u : 65536u + 512u;
      for (int j = 0; j < nch; ++j) {
        const int st = j & 1;
        if (j >= 2 && !mbar_wait_cycles(&bar_empty[st], (uint32_t)((j >> 1) - 1) & 1u, a.err)) {
          abort_flag = 1;
          break;
        }
        uint8_t *stg = sm + st * ST_BYTES;
        const uint8_t *rec = krec(a, s, j, hh);
        mbar_arrive_expect_tx(&bar_full[st], bytes);
        if (half) {
          bulk_load(stg, rec, KR_GC, &bar_full[st]);  // Wk^T, -A diag(b), Khat
          const int rowt = (int)(beg + (int64_t)j * C);
          tma_load_2d(stg + ST_V, &mapV, &bar_full[st], h * D, rowt);
          tma_load_2d(stg + ST_V + 8192, &mapV, &bar_full[st], h * D + 64, rowt);
        } else {
          bulk_load(stg + KR_WH, rec + KR_WH, 32768, &bar_full[st]);
          bulk_load(stg + KR_KH, rec + KR_KH, 32768, &bar_full[st]);
        }
        bulk_load(stg + ST_GC, rec + KR_GC, 512, &bar_full[st]);
      }
    }
    __syncwarp();
  } else if (warp == 8) {
    // ----------------------------------------------------------------------------- MMA warp
    if (lane == 0) {
      const uint32_t id_u = idesc_f32acc(1, 1, 1, 0, 128, 64);   // A = V^T (MN-major), B K-major
      const uint32_t id_p = idesc_f32acc(1, 1, 0, 1, 128, 64);   // A = X^T pieces, B = Wk^T (MN-major)
      const uint32_t id_x = idesc_f32acc(1, 1, 0, 1, 128, 128);  // A = R^T pieces, B = Khat (MN-major)
      constexpr uint64_t DST = ST_BYTES >> 4;
      const uint64_t dV = sdesc_sw128(sb + ST_V, 8192, 1024);
      const uint64_t dAVH = sdesc_sw128(sb + KR_AVH, 16, 1024);
      const uint64_t dAVL = sdesc_sw128(sb + KR_AVL, 16, 1024);
      const uint64_t dWH = sdesc_sw128(sb + KR_WH, 16384, 1024);
      const uint64_t dWL = sdesc_sw128(sb + KR_WL, 16384, 1024);
      const uint64_t dKH = sdesc_sw128(sb + KR_KH, 8192, 1024);
      const uint64_t dKL = sdesc_sw128(sb + KR_KL, 8192, 1024);
      // waits for chunk j's copies; for the S half also issues -U^T of chunk j into P^T (it follows
      // the previous chunk's update in the pipe, which has read the R^T pieces stored there)
      auto stage_ready = [&](int j) -> bool {
        const int st = j & 1;
        if (!mbar_wait_cycles(&bar_full[st], ((uint32_t)j >> 1) & 1u, a.err)) return false;
        tc_fence_after();
        if (half) {
          const uint64_t so = st ? DST : 0;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t av = dV + so + kk * 128;
            mma_f16(tmem + TP, av, dAVH + so + kk * 2, id_u, kk > 0);
            mma_f16(tmem + TP, av, dAVL + so + kk * 2, id_u, 1);
          }
        }
        return true;
      };
      bool ok = stage_ready(0);
      for (int j = 0; j < nch && ok; ++j) {
        const uint64_t so = (j & 1) ? DST : 0;
        const uint32_t par = (uint32_t)j & 1u;
        // P^T in two halves of the contraction, each as soon as its column block is split:
        // block b holds rows i in [32 b, 32 b + 32) and [64 + 32 b, 96 + 32 b), so k-steps
        // {0, 1, 4, 5} then {2, 3, 6, 7}
#pragma unroll
        for (int blk = 0; blk < 2; ++blk) {
          if (!(ok = mbar_wait_cycles(&bar_r1[blk], par, a.err))) break;
          tc_fence_after();
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int kk = 2 * blk + (q & 1) + 4 * (q >> 1);
            const uint64_t wh = dWH + so + kk * 128;
            const uint64_t wl = dWL + so + kk * 128;
            mma_f16_tmem_a(tmem + TP, tmem + TXH + kk * 8, wh, id_p, (half == 1 || blk > 0 || q > 0) ? 1u : 0u);
            mma_f16_tmem_a(tmem + TP, tmem + TXH + kk * 8, wl, id_p, 1);
            mma_f16_tmem_a(tmem + TP, tmem + TXL + kk * 8, wh, id_p, 1);
          }
        }
        if (!ok) break;
        mma_commit(&bar_p);
        if (!(ok = mbar_wait_cycles(&bar_r2, par, a.err))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t bkh = dKH + so + kk * 128;
          const uint64_t bkl = dKL + so + kk * 128;
          const uint32_t pc = tmem + TP + 32 * (kk >> 1) + 8 * (kk & 1);
          mma_f16_tmem_a(tmem + TX, pc, bkh, id_x, 1);
          mma_f16_tmem_a(tmem + TX, pc, bkl, id_x, 1);
          mma_f16_tmem_a(tmem + TX, pc + 16, bkh, id_x, 1);
        }
        // The update's completion frees the state for the next split and this stage for the next
        // copy; the next chunk's U products (S half) follow them, so the split does not wait for U.
        mma_commit(&bar_x);
        mma_commit(&bar_empty[j & 1]);
        if (j + 1 < nch && !(ok = stage_ready(j + 1))) break;
      }
      if (!ok) abort_flag = 1;
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------------ conversion warps
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tx = tmem + lane_base + TX, txh = tmem + lane_base + TXH, txl = tmem + lane_base + TXL;
    const uint32_t tp = tmem + lane_base + TP;
    // X^T = I (T half) or 0 (S half), this thread's columns
    for (int c0 = 64 * part; c0 < 64 * part + 64; c0 += 16) {
      float v[16];
#pragma unroll
      for (int q = 0; q < 16; ++q) v[q] = (half == 0 && c0 + q == row) ? 1.f : 0.f;
      tmem_st16(tx + c0, v);
    }
    tmem_st_wait();
    bool ok = true;
    for (int j = 0; j < nch; ++j) {
      const int st = j & 1;
      const uint32_t par = (uint32_t)j & 1u;
      if (j > 0 && !(ok = mbar_wait_sleep(&bar_x, par ^ 1u, a.err))) break;  // previous update done
      if (!(ok = mbar_wait_sleep(&bar_full[st], ((uint32_t)j >> 1) & 1u, a.err))) break;
      tc_fence_after();
      const float *gC = reinterpret_cast<const float *>(sm + st * ST_BYTES + ST_GC);
      // (1) this thread's 64 rows i of X^T: hi and lo pieces to TMEM, X^T diag(Gamma_C) back.
#pragma unroll
      for (int cb = 0; cb < 64; cb += 32) {
        float xv[32];
        tmem_ld32(tx + 64 * part + cb, xv);
        float ph[16], pl[16];
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          uint32_t hi2, lo2;
          ksplit2(xv[2 * q], xv[2 * q + 1], hi2, lo2);
          ph[q] = __uint_as_float(hi2);
          pl[q] = __uint_as_float(lo2);
        }
        tmem_st16(txh + (64 * part + cb) / 2, ph);
        tmem_st16(txl + (64 * part + cb) / 2, pl);
#pragma unroll
        for (int q = 0; q < 32; ++q) xv[q] *= gC[64 * part + cb + q];
        tmem_st32(tx + 64 * part + cb, xv);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bar_r1[cb / 32]);
      }
      // (2) R^T = -(P^T - U^T): this thread's tokens [32 part, 32 part + 32) as 16 hi then 16 lo columns.
      if (!(ok = mbar_wait_sleep(&bar_p, par, a.err))) break;
      tc_fence_after();
      {
        float pv[32];
        tmem_ld32(tp + 32 * part, pv);
        float ph[16], pl[16];
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          uint32_t hi2, lo2;
          ksplit2(-pv[2 * q], -pv[2 * q + 1], hi2, lo2);
          ph[q] = __uint_as_float(hi2);
          pl[q] = __uint_as_float(lo2);
        }
        tmem_st16(tp + 32 * part, ph);
        tmem_st16(tp + 32 * part + 16, pl);
        tmem_st_wait();
      }
      tc_fence_before();
      mbar_arrive(&bar_r2);
    }
    if (ok && (ok = mbar_wait_cycles(&bar_x, (uint32_t)(nch - 1) & 1u, a.err))) {
      tc_fence_after();
      for (int cb = 0; cb < 64; cb += 32) {
        float xv[32];
        tmem_ld32(tx + 64 * part + cb, xv);
#pragma unroll
        for (int q = 0; q < 32; ++q) out[(size_t)(64 * part + cb + q) * D + row] = xv[q];
      }
    }
    if (!ok) abort_flag = 1;
  }
  __syncthreads();
  tc_fence_after();
  if (abort_flag && tid == 0) {
    // Let any copy or MMA still in flight land before the tensor memory is released.
    for (int k = 0; k < 2; ++k) {
      mbar_wait_cycles(&bar_x, (uint32_t)k, nullptr, 100000000LL);
      mbar_wait_cycles(&bar_p, (uint32_t)k, nullptr, 100000000LL);
      for (int i = 0; i < 2; ++i) {
        mbar_wait_cycles(&bar_full[i], (uint32_t)k, nullptr, 100000000LL);
        mbar_wait_cycles(&bar_empty[i], (uint32_t)k, nullptr, 100000000LL);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

size_t kda_bytes_per_head(int n_seg, int64_t max_len) {
  const int64_t chunks = (max_len + C - 1) / C;
  return (size_t)n_seg * (size_t)(chunks > 0 ? chunks : 1) * KR_REC;
}

}  // namespace

bool build_kda_tc_supported(int D_, int fam, int in_dtype, bool want_o) {
  return D_ == D && in_dtype == HYPIC_BF16 && fam == HYPIC_FAM_KDA && !want_o;
}

size_t build_kda_tc_min_workspace(int n_seg, int64_t max_len) { return kda_bytes_per_head(n_seg, max_len); }

size_t build_kda_tc_workspace_bytes(int H, int n_seg, int64_t max_len) {
  if (H <= 0 || n_seg <= 0) return 0;
  const size_t per = kda_bytes_per_head(n_seg, max_len);
  size_t heads = KWS_CAP / per;
  if (heads < 1) heads = 1;
  if (heads > (size_t)H) heads = (size_t)H;
  return heads * per;
}

// Prep then the chain (both halves in one grid) for each block of heads that fits the workspace.
cudaError_t launch_build_kda_tc(const RecurrentArgs &r, void *ws, size_t ws_bytes, cudaStream_t st) {
  const size_t per = kda_bytes_per_head(r.n_seg, r.seg.max_len);
  const int hb_max = (int)((ws_bytes / per) < (size_t)r.H ? ws_bytes / per : (size_t)r.H);
  if (hb_max < 1 || ws == nullptr) return cudaErrorMemoryAllocation;
  const int nblk = (r.H + hb_max - 1) / hb_max;
  const int Hb = (r.H + nblk - 1) / nblk;
  KdaArgs a{};
  a.H = r.H;
  a.n_seg = r.n_seg;
  a.bounds = r.seg.bounds;
  a.len0 = r.seg.bounds ? 0 : r.seg.uni_len;
  a.max_len = r.seg.max_len;
  a.n_tokens = r.seg.n_tokens < 0 ? INT64_MAX : r.seg.n_tokens;
  a.max_chunks = (int)((r.seg.max_len + C - 1) / C);
  if (a.max_chunks < 1) a.max_chunks = 1;
  a.alpha = r.src.alpha;
  a.beta = r.src.beta;
  a.T_out = r.T_out;
  a.S_out = r.S_out;
  a.ws = static_cast<uint8_t *>(ws);
  a.err = r.err;
  const uint64_t n_tok = r.seg.n_tokens < 0 ? (uint64_t)1 << 31 : (uint64_t)r.seg.n_tokens;
  CUtensorMap mk, mv;
  if (!make_tmap_bf16_2d(&mk, r.src.k, n_tok, (uint64_t)r.H * D, (uint64_t)r.H * D, 64, 64))
    return cudaErrorInvalidValue;
  if (!make_tmap_bf16_2d(&mv, r.src.v, n_tok, (uint64_t)r.H * D, (uint64_t)r.H * D, 64, 64))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(kda_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, KP_SMEM);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(chain_kda_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, KC_SMEM);
  if (e != cudaSuccess) return e;
  for (int h0 = 0; h0 < r.H; h0 += Hb) {
    a.h0 = h0;
    a.Hb = (r.H - h0) < Hb ? (r.H - h0) : Hb;
    const long long g1 = (long long)r.n_seg * a.max_chunks * a.Hb;
    const long long g2 = 2LL * r.n_seg * a.Hb;
    if (g1 > 0x7fffffffLL || g2 > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    kda_prep_kernel<<<(unsigned)g1, NT, KP_SMEM, st>>>(mk, a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    chain_kda_kernel<<<(unsigned)g2, KNT, KC_SMEM, st>>>(mv, a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace hypic
