// Chunked tensor-core segment build for the delta families at d_k = d_v = 128, bf16 inputs.
//
// What it computes (HYPIC reading notes: Method 2 segment pair, paper Sec. 5
// two-pass build, Method 3 Table 3 remark that the delta-type build can use the
// per-step low-rank structure): (T_C, S_{C|0}) of a segment body, as the end
// value of the augmented state X = [T | S] (d_k x 2d) started from [I | 0] and
// run through the gated-delta recurrence with writes only in the S columns.
//
// Chunked (WY) form, 64 tokens per chunk.  With G_t = sum_{r<=t} log a_r inside
// the chunk (kept in base 2 here) and gamma_t = exp(G_t), the per-token rule
//   S_t = a_t S_{t-1} + k_t w_t^T,  w_t^T = b_t (v_t^T - a_t k_t^T S_{t-1})
// unrolls to
//   (I + L) Wm = diag(b) V - diag(b gamma) K X,  L_ts = b_t exp(G_t - G_s) k_t.k_s (s < t)
//   X_new      = gamma_C X + K^T diag(exp(G_C - G_t)) Wm.
// With A = (I + L)^{-1}: Wm = U - Wk X, U = A diag(b) V, Wk = A diag(b gamma) K.
//
// Two kernels per block of heads:
//   wy_prep_kernel  (one CTA per chunk and head, all chunks in parallel): the
//     state-independent part.  TMA loads K; gates and their log-cumsum; Gram =
//     K K^T on tcgen05 (M = 64); L; A = (I + L)^{-1} in fp32, blocked in two levels
//     (16 x 16 diagonal blocks by forward substitution, then 32 x 32); Wk^T = K^T (A diag(b gamma))^T on tcgen05 (K exact in
//     bf16, A diag(b gamma) split hi + lo).  Stored to the workspace as ready-made
//     128-byte-swizzled operand tiles: Wk^T hi + lo, -A diag(b) hi + lo, and the
//     per-token scales exp(G_C - G_t) and gamma_C.
//   chain_tc_kernel (one CTA per segment and head, or at most one CTA per SM running an
//     equal share of all chunk steps, segments cut between CTAs rejoined by composing
//     their pieces' pairs): the state-dependent chain.  The
//     CTA keeps both 128 x 128 fp32 column halves of X (T and S, which evolve
//     independently) in tensor memory for the whole segment, transposed.  Per chunk:
//     TMA brings K, V and the chunk's record (double buffered); -U^T = V^T (-A diag(b))^T
//     goes into the S half's P accumulator; each half splits X^T into bf16 hi (tensor
//     memory) + lo (shared memory) and writes gamma_C X^T back; P^T = X^T Wk^T
//     (hi.hi + hi.lo + lo.hi); R^T = (U^T - P^T) diag(exp(G_C - G_t)) split hi + lo in
//     place; X^T += R^T K.  The two halves run a half-step apart, so one half's
//     conversions overlap the other half's MMAs.
// Operands are fp32-accurate to about 2^-16 relative (bf16 hi + lo; K and V are
// exact in bf16) and every product accumulates in fp32 in TMEM.  Padded tokens of
// a ragged last chunk get b = 0 and a = 1, which makes them exact identity steps.
#include <cuda_bf16.h>

#include <mutex>
#include <type_traits>

#include "tc_ptx.cuh"
#include "tma_host.h"

namespace hypic {
namespace {

using namespace tc;

constexpr int C = 64;    // tokens per chunk
constexpr int D = 128;   // d_k = d_v
constexpr int NT = 128;  // threads per CTA

// Workspace record of one (chunk, head): Wk^T hi and lo as MN-major [128 i][64 t] tiles
// (16 KB each), -A diag(b) hi and lo as K-major [64 t][64 s] tiles (8 KB each), then the
// 65 scales (exp(G_C - G_t) for t < 64, gamma_C), padded.
constexpr uint32_t WS_WH = 0, WS_WL = 16384, WS_AVH = 32768, WS_AVL = 40960, WS_SC = 49152;
constexpr uint32_t WS_TILES = 49152;  // the four tiles, contiguous
constexpr uint32_t WS_SC_BYTES = 272;  // 65 floats rounded up to 16 bytes
constexpr uint32_t WS_REC = 49664;  // bytes per (chunk, head)
// With per-token outputs the record also holds gamma_t = exp(G_t) (64 floats after the scales)
// and the intra-chunk matrix M_ts = exp(G_t - G_s) q_t.k_s (s <= t) as hi and lo K-major
// [64 t][64 s] tiles.
constexpr uint32_t WS_GAM = WS_SC + 272;     // 64 floats
constexpr uint32_t WS_SCG_BYTES = 528;       // scales, gamma_C, padding, gamma_t
constexpr uint32_t WS_MH = 50176, WS_ML = WS_MH + 8192;
constexpr uint32_t WS_REC_O = WS_ML + 8192;  // 66,560
constexpr size_t WS_CAP = (size_t)4 << 30;  // preferred workspace size bound

struct BuildTcArgs {
  int H;       // heads of the token tensors
  int h0, Hb;  // this launch covers heads [h0, h0 + Hb)
  int n_seg;
  const int64_t *bounds;  // [n_seg][2] or null: single segment [0, len0)
  int64_t len0, max_len, n_tokens;
  int max_chunks;
  int fam;
  const float *alpha, *beta;
  float *T_out, *S_out;
  float *o_out;  // [tokens, H, D] or null
  uint8_t *ws;
  uint32_t rec_bytes;  // WS_REC, or WS_REC_O with outputs
  int *err;
  // chain schedule: n_units = n_seg * Hb units of max_chunks steps, q_steps steps per chain CTA;
  // with q_steps > max_chunks, per-CTA pair slots, their publish flags and the CTAs' schedule
  // (both written by the prep kernel)
  int n_units, q_steps, n_flags;
  float *part;
  int *flags;
  int *sched;  // per chain CTA: its chunk steps, then 1 (ends on a cut unit's head) | 2 (bad bounds)
};

__device__ __forceinline__ bool seg_bounds(const BuildTcArgs &a, int s, int64_t &beg, int64_t &end) {
  if (a.bounds) {
    beg = a.bounds[2 * s];
    end = a.bounds[2 * s + 1];
  } else {
    beg = 0;
    end = a.len0;
  }
  return beg >= 0 && end >= beg && end - beg <= a.max_len && end <= a.n_tokens;
}

__device__ __forceinline__ uint8_t *ws_rec(const BuildTcArgs &a, int s, int c, int hh) {
  return a.ws + (((size_t)s * a.max_chunks + c) * a.Hb + hh) * a.rec_bytes;
}

// Work of one chain CTA: the chunk steps [lo, hi) of a list that runs through the units (segment,
// head) in order, max_chunks steps per unit (steps past a segment's end are empty).  With
// q_steps == max_chunks each CTA owns one whole unit.  Otherwise (a grid of at most one CTA per
// SM, launched cooperatively so that all CTAs are resident together) a unit may be cut between
// CTAs b, b + 1, ..., b + m: each later CTA runs its piece of the unit first (the whole of its
// share, for a middle piece) from [I | 0] and publishes the pair in its slot; CTA b runs the
// unit's head last and composes the m published pairs onto it in order, X <- T_c X + [0 | S_c]
// (the composition law of segment pairs), before writing the unit's result.
enum : int { PIECE_WHOLE = 0, PIECE_HEAD = 1, PIECE_TAIL = 2, PIECE_NONE = 3 };  // TAIL: also middle pieces
struct Piece {
  int s, hh;       // the unit
  int64_t beg;     // first token of its body
  int c_lo, c_hi;  // valid chunks [c_lo, c_hi) in this CTA's share
  int kind;
  int n_fix;       // a head: the later pieces to compose onto it
  bool ok;         // segment bounds valid
};
__device__ __forceinline__ Piece piece_of(const BuildTcArgs &a, long long u, long long lo, long long hi) {
  Piece p;
  p.s = (int)(u / a.Hb);
  p.hh = (int)(u % a.Hb);
  int64_t beg = 0, end = 0;
  p.ok = seg_bounds(a, p.s, beg, end);
  p.beg = beg;
  const int nch = p.ok ? (int)((end - beg + C - 1) / C) : 0;
  const long long u0 = u * a.max_chunks;
  const long long s_lo = lo > u0 ? lo - u0 : 0;
  const long long s_hi = hi - u0 < a.max_chunks ? hi - u0 : a.max_chunks;
  p.c_lo = (int)(s_lo < nch ? s_lo : nch);
  p.c_hi = (int)(s_hi < nch ? s_hi : nch);
  if (s_lo == 0)
    p.kind = s_hi >= nch ? PIECE_WHOLE : PIECE_HEAD;
  else
    p.kind = s_lo < nch ? PIECE_TAIL : PIECE_NONE;
  // CTA b + c holds unit steps [s_hi + (c - 1) q, s_hi + c q): a piece while that starts before nch
  p.n_fix = p.kind == PIECE_HEAD ? (int)((nch - s_hi + a.q_steps - 1) / a.q_steps) : 0;
  return p;
}

// Split chain schedule, written by the prep kernel's first CTA (the chain runs after it): the
// chain CTAs' publish flags cleared, and per chain CTA its number of chunk steps and the number of
// pairs it composes onto a cut unit's head at the end (bit 30: it meets a unit with bad bounds).
// The chain then reads its loop bounds with plain loads.
__device__ __noinline__ void chain_schedule(const BuildTcArgs &a) {
  const long long total = (long long)a.n_units * a.max_chunks;
  for (int b = threadIdx.x; b < a.n_flags; b += blockDim.x) {
    a.flags[b] = 0;
    const long long lo = (long long)b * a.q_steps;
    const long long hi = lo + a.q_steps < total ? lo + a.q_steps : total;
    int J = 0, f = 0;
    for (long long u = lo / a.max_chunks; u * a.max_chunks < hi; ++u) {
      const Piece p = piece_of(a, u, lo, hi);
      J += p.c_hi - p.c_lo;
      f = (f & (1 << 30)) | p.n_fix | (p.ok ? 0 : 1 << 30);  // only the last piece can be a head
    }
    a.sched[2 * b] = J;
    a.sched[2 * b + 1] = f;
  }
}

// hi = bf16(v), lo = bf16(v - hi) for 8 values, packed for one 16-byte store each.
__device__ __forceinline__ void split8(const float *v, uint4 &hi, uint4 &lo) {
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

// ------------------------------------------------------------------------------------------------
// Kernel 1: per (segment, chunk, head) -- gates, Gram, L, A = (I + L)^{-1}, operand tiles.
constexpr int LS = 68;                             // row stride of L (floats): conflict-light, 16-byte rows
constexpr uint32_t P_OFF_K = 0;       // 16 KB K chunk, two [64 t][64 i] boxes
constexpr uint32_t P_OFF_L = 16384;   // fp32 [64][LS]: L, then A in place (lower triangle); T = L21 A11
                                      // in its upper-right block; later the A diag(b gamma) hi, lo tiles
constexpr uint32_t P_OFF_AB = P_OFF_L;  // K-major [64 t][64 s] bf16 tiles, 8 KB each
constexpr uint32_t P_OFF_WT = 0;      // Wk^T hi, lo staged for the store, over K and L once both are consumed
constexpr uint32_t P_SMEM = P_OFF_L + 64 * LS * 4 + 1024;  // + alignment slack
constexpr uint32_t P_OFF_Q = 34816;   // with outputs: 16 KB Q chunk, two [64 t][64 i] boxes
constexpr uint32_t P_SMEM_O = P_OFF_Q + 16384 + 1024;

template <bool WO>
__global__ void __launch_bounds__(NT, WO ? 4 : 6)
    wy_prep_kernel(const __grid_constant__ CUtensorMap mapK, const __grid_constant__ CUtensorMap mapQ,
                   const __grid_constant__ BuildTcArgs a) {
  constexpr uint32_t TCOLS = WO ? 128 : 64;  // Gram (and Q K^T at column 64)
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar_tma, bar_mma;
  __shared__ uint32_t tmem_slot;
  __shared__ float sG[C], sBv[C], sBG[C];
  __shared__ int ok_flag;
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float *sL = reinterpret_cast<float *>(sm + P_OFF_L);
  float *sA = sL;  // A = (I + L)^{-1} replaces L in place, row stride LS
  float *sT = sL + 32;  // [32][32] with row stride LS: rows 0..31, columns 32..63 of L (never read as L)
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  if (blockIdx.x == 0 && a.flags) chain_schedule(a);
  const int hh = blockIdx.x % a.Hb;
  const int c = (blockIdx.x / a.Hb) % a.max_chunks;
  const int s = (blockIdx.x / a.Hb) / a.max_chunks;
  const int h = a.h0 + hh;
  int64_t beg, end;
  if (!seg_bounds(a, s, beg, end)) return;  // reported by the chain kernel
  if ((int64_t)c * C >= end - beg) return;
  const int64_t t0 = beg + (int64_t)c * C;

  if (tid == 0) {
    mbar_init(&bar_tma, 1);
    mbar_init(&bar_mma, 1);
    mbar_fence_init();
    ok_flag = 1;
    mbar_arrive_expect_tx(&bar_tma, WO ? 32768 : 16384);
    tma_load_2d(sm + P_OFF_K, &mapK, &bar_tma, h * D, (int)t0);
    tma_load_2d(sm + P_OFF_K + 8192, &mapK, &bar_tma, h * D + 64, (int)t0);
    if (WO) {
      tma_load_2d(sm + P_OFF_Q, &mapQ, &bar_tma, h * D, (int)t0);
      tma_load_2d(sm + P_OFF_Q + 8192, &mapQ, &bar_tma, h * D + 64, (int)t0);
    }
  }
  if (warp == 0) {
    tmem_alloc(&tmem_slot, TCOLS);
    tmem_relinquish();
  }
  // gates: G_t = inclusive log2-cumsum of a, masked beyond the body
  if (tid < C) {
    const int64_t tok = t0 + tid;
    float av = 1.f, bv = 0.f;
    if (tok < end) {
      bv = a.beta[tok * a.H + h];
      if (a.fam == HYPIC_FAM_GATED_DELTA) av = a.alpha[tok * a.H + h];
    }
    float g = log2f(av);
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, g, o);
      if (lane >= o) g += y;
    }
    sG[tid] = g;
    sBv[tid] = bv;
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  if (tid >= 32 && tid < C) sG[tid] += sG[31];
  if (tid == 0) {
    if (!mbar_wait_cycles(&bar_tma, 0, a.err)) ok_flag = 0;
    if (ok_flag) {
      const uint32_t kb = smem_u32(sm + P_OFF_K);
      const uint32_t id = idesc_f32acc(1, 1, 0, 0, 64, 64);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint32_t off = (kk >> 2) * 8192 + (kk & 3) * 32;
        mma_f16(tmem, sdesc_sw128(kb + off, 16, 1024), sdesc_sw128(kb + off, 16, 1024), id, kk > 0);
      }
      if (WO) {
        // Q K^T (M = 64 t, N = 64 s, K = 128 i), Q and K exact in bf16
        const uint32_t qb = smem_u32(sm + P_OFF_Q);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk >> 2) * 8192 + (kk & 3) * 32;
          mma_f16(tmem + 64, sdesc_sw128(qb + off, 16, 1024), sdesc_sw128(kb + off, 16, 1024), id, kk > 0);
        }
      }
      mma_commit(&bar_mma);
      if (!mbar_wait_cycles(&bar_mma, 0, a.err)) ok_flag = 0;
    }
  }
  // Decay factors: 2^(G_t - G_s) = e_t f_s with e_t = 2^(G_t - G_m), f_s = 2^(G_m - G_s) around the
  // middle token m, exact in fp32 while the chunk's total log2-decay stays within 100 (gates
  // averaging above 0.33 per token); otherwise every factor is taken as one exponential.
  __shared__ float sE[C], sF[C];
  __syncthreads();
  tc_fence_after();
  const bool separable = (sG[0] - sG[C - 1]) < 100.f;
  if (tid < C) {
    sBG[tid] = sBv[tid] * exp2f(sG[tid]);
    sE[tid] = exp2f(sG[tid] - sG[C / 2]);
    sF[tid] = exp2f(sG[C / 2] - sG[tid]);
  }
  __syncthreads();
  if (ok_flag) {
    // L_ts = b_t 2^(G_t - G_s) Gram_ts (s < t).  Gram row t sits in lane 32 (t / 16) + t % 16; the
    // 16x256b load spreads a warp's 16 rows over all its threads: rows ta and ta + 8, two columns
    // of each group of eight.
    const int ta = warp * 16 + (lane >> 2), tb = ta + 8, cq = 2 * (lane & 3);
    float v[32];
    tmem_ld16x256_x8(tmem + ((uint32_t)(warp * 32) << 16), v);
    if (separable) {
      const float ea = sBv[ta] * sE[ta], eb = sBv[tb] * sE[tb];
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        const int sc = 8 * m + cq;
        const float2 f2 = *reinterpret_cast<const float2 *>(sF + sc);
        *reinterpret_cast<float2 *>(sL + ta * LS + sc) =
            make_float2(sc < ta ? ea * f2.x * v[4 * m] : 0.f, sc + 1 < ta ? ea * f2.y * v[4 * m + 1] : 0.f);
        *reinterpret_cast<float2 *>(sL + tb * LS + sc) =
            make_float2(sc < tb ? eb * f2.x * v[4 * m + 2] : 0.f, sc + 1 < tb ? eb * f2.y * v[4 * m + 3] : 0.f);
      }
    } else {
      const float ba = sBv[ta], bb = sBv[tb], Ga = sG[ta], Gb = sG[tb];
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        const int sc = 8 * m + cq;
        const float g0 = sG[sc], g1 = sG[sc + 1];
        *reinterpret_cast<float2 *>(sL + ta * LS + sc) =
            make_float2(sc < ta ? ba * exp2f(Ga - g0) * v[4 * m] : 0.f,
                        sc + 1 < ta ? ba * exp2f(Ga - g1) * v[4 * m + 1] : 0.f);
        *reinterpret_cast<float2 *>(sL + tb * LS + sc) =
            make_float2(sc < tb ? bb * exp2f(Gb - g0) * v[4 * m + 2] : 0.f,
                        sc + 1 < tb ? bb * exp2f(Gb - g1) * v[4 * m + 3] : 0.f);
      }
    }
  }
  if (WO && ok_flag) {
    // M_ts = 2^(G_t - G_s) (Q K^T)_ts for s <= t, split hi + lo into the K-major [t][s] tiles of
    // the record; gamma_t = 2^(G_t).
    uint8_t *rec = ws_rec(a, s, c, hh);
    const int t = warp * 16 + lane;
    const float et = lane < 16 ? sE[t] : 0.f;
    const float Gt = lane < 16 ? sG[t] : 0.f;
#pragma unroll 1
    for (int hb = 0; hb < C; hb += 32) {
      float v[32];
      tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + 64 + hb, v);
      if (lane < 16) {
#pragma unroll
        for (int q = 0; q < 32; q += 8) {
          float m8[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int sc = hb + q + e;
            const float dec = separable ? et * sF[sc] : exp2f(Gt - sG[sc]);
            m8[e] = sc <= t ? dec * v[q + e] : 0.f;
          }
          uint4 hi, lo;
          split8(m8, hi, lo);
          const uint32_t off = sw128_offset((uint32_t)t, (uint32_t)((hb + q) >> 3));
          *reinterpret_cast<uint4 *>(rec + WS_MH + off) = hi;
          *reinterpret_cast<uint4 *>(rec + WS_ML + off) = lo;
        }
      }
    }
    if (tid < C) reinterpret_cast<float *>(rec + WS_GAM)[tid] = exp2f(sG[tid]);
  }
  tc_fence_before();
  __syncthreads();
  if (!ok_flag) {
    if (warp == 0) tmem_dealloc(tmem, TCOLS);
    return;
  }

  // Diagonal 16 x 16 blocks of A by column-wise forward substitution (threads 0..63, one column
  // each), written over the blocks of L they came from once every thread has read them.
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
  // Lower-left 16 x 16 quarter of each diagonal 32 x 32 block p (16-blocks a = 2p, b = 2p + 1):
  // A_ba = -A_bb (L_ba A_aa).  Thread -> block p = tid / 64, row tid % 64 / 4, four columns; the
  // product L_ba A_aa waits in the free upper-right region (rows 0..15, columns 32 + 16 p ..).
  {
    const int p = tid >> 6, r = (tid & 63) >> 2, c0 = 4 * (tid & 3);
    const int o = 32 * p;  // the 32-block's first row and column
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
    float *Y = sT + 16 * p;  // rows 0..15, columns 32 + 16 p + 0..15 of L's frame
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
  // T = L21 A11 and A21 = -A22 T (32 x 32 each): each thread owns a 2 x 4 output tile
  // (rows 2 (tid / 8) + {0, 1}, columns 4 (tid % 8) + {0..3}).
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
    // A22 is lower triangular: rows r0, r0 + 1 of warp w (rows 8 w .. 8 w + 7) need k < 8 w + 8.
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

  // Operand tiles, split hi + lo, 128-byte-swizzled K-major [64 t][64 s]: -A diag(b) straight to
  // the workspace record; A diag(b gamma) into shared memory (over A, once all of A is read) for
  // the Wk^T product.  Entries above the diagonal of A are zero (the upper-right block holds T).
  uint8_t *rec = ws_rec(a, s, c, hh);
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
      vb[i] = av * sBG[8 * q + i];
      vv[i] = -av * sBv[8 * q + i];  // negated: the chain accumulates -U under P
    }
    uint4 hi, lo;
    const uint32_t off = sw128_offset((uint32_t)t, (uint32_t)q);
    split8(vb, abh[j], abl[j]);
    split8(vv, hi, lo);
    *reinterpret_cast<uint4 *>(rec + WS_AVH + off) = hi;
    *reinterpret_cast<uint4 *>(rec + WS_AVL + off) = lo;
  }
  __syncthreads();
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int e = tid + j * NT;
    const uint32_t off = sw128_offset((uint32_t)(e >> 3), (uint32_t)(e & 7));
    *reinterpret_cast<uint4 *>(sm + P_OFF_AB + off) = abh[j];
    *reinterpret_cast<uint4 *>(sm + P_OFF_AB + 8192 + off) = abl[j];
  }
  float *sc = reinterpret_cast<float *>(rec + WS_SC);
  if (tid < C) sc[tid] = exp2f(sG[C - 1] - sG[tid]);
  if (tid == 0) sc[C] = exp2f(sG[C - 1]);
  fence_proxy_async();
  __syncthreads();

  // Wk^T = K^T (A diag(b gamma))^T: M = 128 (i), N = 64 (t), K = 64 (s), into the Gram's columns.
  if (tid == 0) {
    tc_fence_after();
    const uint32_t kb = smem_u32(sm + P_OFF_K), ab = smem_u32(sm + P_OFF_AB);
    const uint32_t id = idesc_f32acc(1, 1, 1, 0, 128, 64);  // A = K^T (MN-major), B K-major
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      const uint64_t ak = sdesc_sw128(kb + kk * 2048, 8192, 1024);
      mma_f16(tmem, ak, sdesc_sw128(ab + kk * 32, 16, 1024), id, kk > 0);
      mma_f16(tmem, ak, sdesc_sw128(ab + 8192 + kk * 32, 16, 1024), id, 1);
    }
    mma_commit(&bar_mma);
    if (!mbar_wait_cycles(&bar_mma, 1, a.err)) ok_flag = 0;
  }
  __syncthreads();
  tc_fence_after();
  if (ok_flag) {
    // lane i = tid holds Wk^T row i: split into the MN-major [128 i][64 t] hi and lo tiles.
#pragma unroll 1
    for (int hb = 0; hb < C; hb += 32) {
      float wv[32];
      tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + hb, wv);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint4 hi, lo;
        split8(wv + 8 * q, hi, lo);
        const uint32_t off = sw128_offset((uint32_t)tid, (uint32_t)(hb / 8 + q));
        *reinterpret_cast<uint4 *>(sm + P_OFF_WT + off) = hi;
        *reinterpret_cast<uint4 *>(sm + P_OFF_WT + 16384 + off) = lo;
      }
    }
  }
  fence_proxy_async();
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, TCOLS);
  if (ok_flag && tid == 0) {
    bulk_store(rec + WS_WH, sm + P_OFF_WT, 32768);
    bulk_store_commit();
    bulk_store_wait_read();  // the shared source must outlive the copy; the CTA may then exit
  }
}

// ------------------------------------------------------------------------------------------------
// Kernel 2: per (segment, head) -- the chunk chain of both column halves on tensor memory.
//
// Each half's state is kept transposed, X^T (lanes = the 128 columns n of the half, TMEM columns
// = rows i), so that both state-dependent products take their A operand from tensor or shared
// memory and read only their B operand from the chunk's tiles:
//   P^T - U^T = X^T Wk^T - U^T   A = X^T hi (TMEM) / lo (shared), B = Wk^T [i][t] (MN-major)
//   X^T = gamma_C X^T + R^T K    A = R^T hi/lo pieces (TMEM, in place over P^T), B = K [t][i]
// -U^T = V^T (-A diag(b))^T is written into the S half's P accumulator first.  Warp 16 issues
// every MMA, warp 17 every TMA copy; warps 0-7 convert for the T half and warps 8-15 for the S
// half (two threads per TMEM lane each).  MMA completions reach the converters through tcgen05.commit;
// the converters arrive after their TMEM and shared-memory writes are fenced.
constexpr uint32_t STAGE_K = 0, STAGE_V = 16384, STAGE_REC = 32768;  // within a stage
constexpr uint32_t STAGE_BYTES = STAGE_REC + WS_TILES;               // 81,920 (1024-aligned)
constexpr uint32_t OFF_XLO = 2 * STAGE_BYTES;                        // X^T lo tiles, 32 KB per half
constexpr uint32_t OFF_SC = OFF_XLO + 65536;                         // scales, 512 B per stage
constexpr uint32_t SMEM_BYTES = OFF_SC + 1024 + 1024;                // + alignment slack

// Tensor memory (512 columns): per half h, X^T at 128 h, X^T hi pieces at 256 + 64 h, P^T (then
// the R^T pieces) at 384 + 64 h.
__device__ __forceinline__ uint32_t tm_x(int h) { return 128u * h; }
__device__ __forceinline__ uint32_t tm_xp(int h) { return 256u + 64u * h; }
__device__ __forceinline__ uint32_t tm_p(int h) { return 384u + 64u * h; }
constexpr uint32_t TM_COLS = 512;

constexpr int NCONV = 512;       // conversion threads: two per TMEM lane and half
constexpr int NT2 = NCONV + 64;  // + the MMA warp and the TMA warp

// hi = truncation of x to bf16, lo = bf16 rounding of the exact remainder, for two values;
// returns the packed hi pair and lo pair (first value in the low half).
__device__ __forceinline__ void split2_pair(float a, float b, uint32_t &hi, uint32_t &lo) {
  const uint32_t ua = __float_as_uint(a), ub = __float_as_uint(b);
  const float ra = a - __uint_as_float(ua & 0xFFFF0000u), rb = b - __uint_as_float(ub & 0xFFFF0000u);
  hi = __byte_perm(ua, ub, 0x7632);
  const __nv_bfloat162 lp = __floats2bfloat162_rn(ra, rb);
  lo = *reinterpret_cast<const uint32_t *>(&lp);
}

// This CTA's step range [lo, hi).
__device__ __forceinline__ void cta_steps(const BuildTcArgs &a, long long &lo, long long &hi) {
  const long long total = (long long)a.n_units * a.max_chunks;
  lo = (long long)blockIdx.x * a.q_steps;
  hi = lo + a.q_steps < total ? lo + a.q_steps : total;
}
// The piece of unit u in this CTA's share.  Piece walks run where a piece starts or ends, so they
// are kept out of line, away from the code of the chunk loops.
__device__ __noinline__ Piece piece_at(const BuildTcArgs &a, int u) {
  long long lo, hi;
  cta_steps(a, lo, hi);
  return piece_of(a, u, lo, hi);
}
__device__ __noinline__ int units_begin(const BuildTcArgs &a) {
  long long lo, hi;
  cta_steps(a, lo, hi);
  return (int)(lo / a.max_chunks);
}
__device__ __noinline__ int units_end(const BuildTcArgs &a) {
  long long lo, hi;
  cta_steps(a, lo, hi);
  return (int)((hi + a.max_chunks - 1) / a.max_chunks);
}
// The first unit from u on with chunks in this CTA's share (units_end if none).
__device__ __noinline__ int next_busy_unit(const BuildTcArgs &a, int u) {
  const int ue = units_end(a);
  for (; u < ue; ++u) {
    const Piece p = piece_at(a, u);
    if (p.c_hi > p.c_lo) break;
  }
  return u;
}

__device__ __forceinline__ void st_release_gpu(int *f, int v) {
  asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(f), "r"(v) : "memory");
}
// Waits (bounded) for a neighbour's published pair: true if it was published intact.
__device__ __forceinline__ bool wait_published(const int *f, int *err, long long limit = 2000000000LL) {
  const long long t0 = clock64();
  for (;;) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(f) : "memory");
    if (v != 0) return v == 1;
    if (clock64() - t0 > limit) {
      set_error(err, HYPIC_ETIMEOUT);
      return false;
    }
    __nanosleep(200);
  }
}

// The composition of a cut unit stages T_B as bf16 hi and lo K-major tiles ([128 i][64 j] blocks
// of 16 KB) in stage 0, which no chunk uses any more by then.
constexpr uint32_t FX_TBH = 0, FX_TBL = 32768;

// ---- conversion-thread helpers (thread t < 512: TMEM lane t & 127, column part (t >> 7) & 1,
// half (t >> 8) & 1) --------------------------------------------------------------------------
__device__ __forceinline__ int conv_row() { return threadIdx.x & 127; }
__device__ __forceinline__ int conv_part() { return (threadIdx.x >> 7) & 1; }
__device__ __forceinline__ int conv_half() { return (threadIdx.x >> 8) & 1; }

// X^T = [I | 0]^T restricted to this thread's half and columns: I (T half) or 0 (S half).
__device__ __noinline__ void conv_init_x(uint32_t tx) {
  const int row = conv_row(), part = conv_part(), half = conv_half();
  for (int c0 = 64 * part; c0 < 64 * part + 64; c0 += 16) {
    float v[16];
#pragma unroll
    for (int q = 0; q < 16; ++q) v[q] = (half == 0 && c0 + q == row) ? 1.f : 0.f;
    tmem_st16(tx + c0, v);
  }
  tmem_st_wait();
}
// Copies this thread's 64 rows i of its half's X^T to out[i][n] (row-major [128][128]).
__device__ __noinline__ void conv_write_x(uint32_t tx, float *out) {
  const int row = conv_row(), part = conv_part();
  for (int cb = 0; cb < 64; cb += 32) {
    float xv[32];
    tmem_ld32(tx + 64 * part + cb, xv);
#pragma unroll
    for (int q = 0; q < 32; ++q) out[(size_t)(64 * part + cb + q) * D + row] = xv[q];
  }
}
__device__ __forceinline__ float *unit_out(const BuildTcArgs &a, const Piece &p, int half) {
  return (half ? a.S_out : a.T_out) + ((size_t)p.s * a.H + a.h0 + p.hh) * D * D;
}
// Units of this CTA with no chunks to run: empty bodies get [I | 0]; cuts past a body's end leave
// nothing to do.
__device__ __noinline__ void conv_empty_units(const BuildTcArgs &a) {
  const int row = conv_row(), part = conv_part(), half = conv_half();
  const int ue = units_end(a);
  for (int u = units_begin(a); u < ue; ++u) {
    const Piece p = piece_at(a, u);
    if (p.kind != PIECE_WHOLE || p.c_hi > p.c_lo) continue;
    float *out = unit_out(a, p, half);
    for (int i = 64 * part; i < 64 * part + 64; ++i) out[(size_t)i * D + row] = (half == 0 && i == row) ? 1.f : 0.f;
  }
}
// A cut unit's tail: publish (T_B, S_B) for the previous CTA, which composes it onto the head.
__device__ __noinline__ void conv_publish(const BuildTcArgs &a, uint32_t tx, bool ok) {
  if (ok) conv_write_x(tx, a.part + ((size_t)blockIdx.x * 2 + conv_half()) * D * D);
  __threadfence();
  const bool bad = bar_or_named(1, NCONV, !ok);
  if (threadIdx.x == 0) st_release_gpu(&a.flags[blockIdx.x], bad ? 2 : 1);
}
// A cut unit's head (this CTA's last piece): stage T_B as the B tiles of X^T += X_A^T T_B^T, split
// X_A^T like step (1) of a chunk, restart the accumulator at [0 | S_B]^T and hand over to the MMA
// warp; then write the unit's result.  Both halves' last updates have landed before the tiles are
// written over stage 0.
__device__ __noinline__ bool conv_compose_head(const BuildTcArgs &a, const Piece &p, uint32_t tx, uint32_t txp,
                                               uint8_t *xlo, uint8_t *sm, uint64_t *bar_r1h, uint64_t *bar_xh,
                                               int J, bool ok) {
  const int tid = threadIdx.x, row = conv_row(), part = conv_part(), half = conv_half();
  bool bad = false;
  for (int c = 1; c <= p.n_fix; ++c) {
    const float *pairB = a.part + (size_t)(blockIdx.x + c) * 2 * D * D;
    if (tid == 0 && ok && !bad) ok = wait_published(&a.flags[blockIdx.x + c], a.err);
    // Past this barrier both halves' previous MMAs are done, so stage 0 is free.
    bad = bar_or_named(1, NCONV, !ok || bad);
    if (!bad) {
      // T_B as K-major bf16 hi and lo tiles: thread -> row i, columns [32 qb, 32 qb + 32).
      const int i = tid >> 2, qb = tid & 3;
      const float *src = pairB + (size_t)i * D + 32 * qb;
      for (int m = 0; m < 4; ++m) {
        float v[8];
        const float4 v0 = __ldcg(reinterpret_cast<const float4 *>(src + 8 * m));
        const float4 v1 = __ldcg(reinterpret_cast<const float4 *>(src + 8 * m + 4));
        v[0] = v0.x; v[1] = v0.y; v[2] = v0.z; v[3] = v0.w;
        v[4] = v1.x; v[5] = v1.y; v[6] = v1.z; v[7] = v1.w;
        uint4 h8, l8;
        split8(v, h8, l8);
        const uint32_t col = 32u * qb + 8u * m;
        const uint32_t off = (col / 64) * 16384u + sw128_offset((uint32_t)i, (col % 64) / 8);
        *reinterpret_cast<uint4 *>(sm + FX_TBH + off) = h8;
        *reinterpret_cast<uint4 *>(sm + FX_TBL + off) = l8;
      }
      // X^T pieces as in step (1); the accumulator restarts at [0 | S_B]^T.
      const float *sB = pairB + (size_t)D * D;
      for (int cb = 0; cb < 64; cb += 32) {
        float xv[32];
        tmem_ld32(tx + 64 * part + cb, xv);
        float ph[16];
        uint32_t pl[16];
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          uint32_t hi2;
          split2_pair(xv[2 * q], xv[2 * q + 1], hi2, pl[q]);
          ph[q] = __uint_as_float(hi2);
        }
        tmem_st16(txp + (64 * part + cb) / 2, ph);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          *reinterpret_cast<uint4 *>(xlo + sw128_offset((uint32_t)row, (uint32_t)(cb / 8 + k))) =
              make_uint4(pl[4 * k], pl[4 * k + 1], pl[4 * k + 2], pl[4 * k + 3]);
#pragma unroll
        for (int q = 0; q < 32; ++q) xv[q] = half ? __ldcg(sB + (size_t)(64 * part + cb + q) * D + row) : 0.f;
        tmem_st32(tx + 64 * part + cb, xv);
      }
      tmem_st_wait();
    }
    fence_proxy_async();
    tc_fence_before();
    bar_sync_named(1, NCONV);  // T_B tiles complete
    mbar_arrive(bar_r1h);
    const bool fx = mbar_wait_sleep(bar_xh, (uint32_t)(J + c - 1) & 1u, a.err);
    tc_fence_after();
    ok = ok && fx;
  }
  ok = ok && !bad;
  if (ok) conv_write_x(tx, unit_out(a, p, half));
  return ok;
}
// The MMA warp's part of a cut unit's head, once per published pair: X^T += X^T T_B^T on top of
// [0 | S_B]^T per half (M = 128 n, N = 128 i, K = 128 j), hi.hi + hi.lo + lo.hi with T_B split like
// the chunk operands.
__device__ __noinline__ bool mma_compose_head(uint32_t tmem, uint32_t sb, uint64_t *bar_r1, uint64_t *bar_x, int J,
                                              int n_fix, int *err) {
  const uint32_t id_f = idesc_f32acc(1, 1, 0, 0, 128, 128);
  const uint64_t dTH = sdesc_sw128(sb + FX_TBH, 16, 1024);
  const uint64_t dTL = sdesc_sw128(sb + FX_TBL, 16, 1024);
  const uint64_t dXL = sdesc_sw128(sb + OFF_XLO, 16, 1024);
  for (int c = 0; c < n_fix; ++c) {
    for (int hf = 0; hf < 2; ++hf) {
      if (!mbar_wait_cycles(&bar_r1[hf], (uint32_t)(J + c) & 1u, err)) return false;
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint64_t ko = (uint64_t)(kk >> 2) * (16384 >> 4) + (kk & 3) * 2;
        const uint64_t al = dXL + hf * 2048 + (kk >> 2) * 1024 + (kk & 3) * 2;
        mma_f16_tmem_a(tmem + tm_x(hf), tmem + tm_xp(hf) + kk * 8, dTH + ko, id_f, 1);
        mma_f16_tmem_a(tmem + tm_x(hf), tmem + tm_xp(hf) + kk * 8, dTL + ko, id_f, 1);
        mma_f16(tmem + tm_x(hf), al, dTH + ko, id_f, 1);
      }
      mma_commit(&bar_x[hf]);
    }
  }
  return true;
}

template <bool T_ONLY>
__global__ void __launch_bounds__(NT2, 1)
    chain_tc_kernel(const __grid_constant__ CUtensorMap mapK, const __grid_constant__ CUtensorMap mapV,
                    const __grid_constant__ BuildTcArgs a) {
  extern __shared__ uint8_t smem_raw[];
  // per half: r1 (X pieces ready), r2 (R pieces ready), p (P^T done), x (update done)
  // per stage: full (copies landed), empty (the chunk's last MMAs done)
  __shared__ uint64_t bar_full[2], bar_empty[2], bar_r1[2], bar_r2[2], bar_p[2], bar_x[2];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(sm);
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const bool issuer = warp == NCONV / 32, producer = warp == NCONV / 32 + 1;
  const int row = tid & 127;        // TMEM lane a conversion thread serves
  const int part = (tid >> 7) & 1;  // which half of that lane's columns
  const int half = (tid >> 8) & 1;  // 0: T columns, 1: S columns

  // This CTA's chunk steps J and the pairs it composes onto a cut unit's head at the end: from the
  // schedule the prep kernel wrote, or with one unit per CTA straight from the unit's bounds.
  int J = 0, n_fix = 0;
  bool bounds_ok = true;
  if (a.sched) {
    J = a.sched[2 * blockIdx.x];
    const int f = a.sched[2 * blockIdx.x + 1];
    n_fix = f & 0xffff;
    bounds_ok = (f & (1 << 30)) == 0;
  } else {
    int64_t beg, end;
    bounds_ok = seg_bounds(a, (int)(blockIdx.x / a.Hb), beg, end);
    J = bounds_ok ? (int)((end - beg + C - 1) / C) : 0;
  }
  if (!bounds_ok) {
    if (tid == 0) {
      set_error(a.err, HYPIC_EDEVICE);
      if (a.flags) st_release_gpu(&a.flags[blockIdx.x], 2);  // a waiting neighbour goes on
    }
    return;
  }

  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar_full[i], 1);
      mbar_init(&bar_empty[i], 1);
      mbar_init(&bar_r1[i], 256);
      mbar_init(&bar_r2[i], 256);
      mbar_init(&bar_p[i], 1);
      mbar_init(&bar_x[i], 1);
    }
    mbar_fence_init();
    abort_flag = 0;
  }
  if (warp == 0) {
    tmem_alloc(&tmem_slot, TM_COLS);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;

  if (producer) {
    // ------------------------------------------------------------------------------- TMA warp
    // Chunk step j goes into stage j & 1 once step j - 2, the stage's previous user, has run its
    // last MMAs (the converters are done with the stage before those are issued).
    if (lane == 0) {
      prefetch_tmap(&mapK);
      prefetch_tmap(&mapV);
      bool ok = true;
      int j = 0;
      const int ue = units_end(a);
      for (int u = units_begin(a); u < ue && ok; ++u) {
        const Piece p = piece_at(a, u);
        const int h = a.h0 + p.hh;
        for (int c = p.c_lo; c < p.c_hi; ++c, ++j) {
          const int st = j & 1;
          if (j >= 2 && !(ok = mbar_wait_cycles(&bar_empty[st], (uint32_t)((j >> 1) - 1) & 1u, a.err))) break;
          const int rowt = (int)(p.beg + (int64_t)c * C);
          uint8_t *stg = sm + st * STAGE_BYTES;
          const uint8_t *rec = ws_rec(a, p.s, c, p.hh);
          mbar_arrive_expect_tx(&bar_full[st], 32768u + WS_TILES + WS_SC_BYTES);
          tma_load_2d(stg + STAGE_K, &mapK, &bar_full[st], h * D, rowt);
          tma_load_2d(stg + STAGE_K + 8192, &mapK, &bar_full[st], h * D + 64, rowt);
          tma_load_2d(stg + STAGE_V, &mapV, &bar_full[st], h * D, rowt);
          tma_load_2d(stg + STAGE_V + 8192, &mapV, &bar_full[st], h * D + 64, rowt);
          bulk_load(stg + STAGE_REC, rec, WS_TILES, &bar_full[st]);
          bulk_load(sm + OFF_SC + st * 512, rec + WS_SC, WS_SC_BYTES, &bar_full[st]);
        }
      }
      if (!ok) abort_flag = 1;
    }
    __syncwarp();
  } else if (issuer) {
    // ------------------------------------------------------------------------------- MMA warp
    if (lane == 0) {
      const uint32_t id_u = idesc_f32acc(1, 1, 1, 0, 128, 64);   // A = V^T (MN-major), B K-major
      const uint32_t id_p = idesc_f32acc(1, 1, 0, 1, 128, 64);   // A = X^T pieces, B = Wk^T (MN-major)
      const uint32_t id_x = idesc_f32acc(1, 1, 0, 1, 128, 128);  // A = R^T pieces (TMEM), B = K
      // Shared-memory descriptors as a base per operand plus constant offsets: the address field
      // holds addr >> 4 in its low 14 bits and no operand crosses 256 KB, so an offset of off
      // bytes adds off >> 4 to the descriptor.
      constexpr uint64_t DSTG = STAGE_BYTES >> 4;
      const uint64_t dV = sdesc_sw128(sb + STAGE_V, 8192, 1024);
      const uint64_t dK = sdesc_sw128(sb + STAGE_K, 8192, 1024);
      const uint64_t dAVH = sdesc_sw128(sb + STAGE_REC + WS_AVH, 16, 1024);
      const uint64_t dAVL = sdesc_sw128(sb + STAGE_REC + WS_AVL, 16, 1024);
      const uint64_t dWH = sdesc_sw128(sb + STAGE_REC + WS_WH, 16384, 1024);
      const uint64_t dWL = sdesc_sw128(sb + STAGE_REC + WS_WL, 16384, 1024);
      const uint64_t dXL = sdesc_sw128(sb + OFF_XLO, 16, 1024);
      // -U^T of step j (in stage st = j & 1) into the S half's P^T (M = 128 j, N = 64 t,
      // K = 64 s).  It follows the previous step's S update in the pipe, which has read the R^T
      // pieces stored there.
      auto issue_u = [&](int j, auto st_tag) -> bool {
        constexpr int st = decltype(st_tag)::value;
        if (!mbar_wait_cycles(&bar_full[st], ((uint32_t)j >> 1) & 1u, a.err)) return false;
        tc_fence_after();
        if (T_ONLY) return true;
        constexpr uint64_t so = st ? DSTG : 0;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t av = dV + so + kk * 128;
          mma_f16(tmem + tm_p(1), av, dAVH + so + kk * 2, id_u, kk > 0);
          mma_f16(tmem + tm_p(1), av, dAVL + so + kk * 2, id_u, 1);
        }
        return true;
      };
      constexpr int nh = T_ONLY ? 1 : 2;
      auto step = [&](const int j) -> bool {
        const int ST = j & 1;
        const uint32_t par = ST;
        const uint64_t so = ST ? DSTG : 0;
#pragma unroll
        for (int hf = 0; hf < nh; ++hf) {
          if (!mbar_wait_cycles(&bar_r1[hf], par, a.err)) return false;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint64_t wh = dWH + so + kk * 128;
            const uint64_t wl = dWL + so + kk * 128;
            const uint64_t al = dXL + hf * 2048 + (kk >> 2) * 1024 + (kk & 3) * 2;
            mma_f16_tmem_a(tmem + tm_p(hf), tmem + tm_xp(hf) + kk * 8, wh, id_p, (hf == 1 || kk > 0) ? 1u : 0u);
            mma_f16_tmem_a(tmem + tm_p(hf), tmem + tm_xp(hf) + kk * 8, wl, id_p, 1);
            mma_f16(tmem + tm_p(hf), al, wh, id_p, 1);
          }
          mma_commit(&bar_p[hf]);
        }
#pragma unroll
        for (int hf = 0; hf < nh; ++hf) {
          if (!mbar_wait_cycles(&bar_r2[hf], par, a.err)) return false;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t bk = dK + so + kk * 128;
            const uint32_t pc = tmem + tm_p(hf) + 32 * (kk >> 1) + 8 * (kk & 1);
            mma_f16_tmem_a(tmem + tm_x(hf), pc, bk, id_x, 1);
            mma_f16_tmem_a(tmem + tm_x(hf), pc + 16, bk, id_x, 1);
          }
          if (hf == nh - 1 && j + 1 < J) {
            const bool r = ST ? issue_u(j + 1, std::integral_constant<int, 0>{}) : issue_u(j + 1, std::integral_constant<int, 1>{});
            if (!r) return false;
          }
          mma_commit(&bar_x[hf]);
        }
        mma_commit(&bar_empty[ST]);
        return true;
      };
      bool ok = J == 0 || issue_u(0, std::integral_constant<int, 0>{});
      for (int j = 0; j < J && ok; ++j) ok = step(j);
      if constexpr (!T_ONLY)
        if (ok && n_fix > 0) ok = mma_compose_head(tmem, sb, bar_r1, bar_x, J, n_fix, a.err);
      if (!ok) abort_flag = 1;
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------------- conversion warps
    const uint32_t tx = tmem + lane_base + tm_x(half), txp = tmem + lane_base + tm_xp(half);
    const uint32_t tp = tmem + lane_base + tm_p(half);
    uint8_t *xlo = sm + OFF_XLO + half * 32768 + part * 16384;
    const bool idle = T_ONLY && half == 1;  // the T-only chain has no S half
    if (!idle) conv_empty_units(a);
    // The current piece and the next busy one stay in registers as a unit index, kind | n_fix << 2
    // and (next) length: the next is looked up during a piece's first step, while its P^T products
    // run, so a piece boundary does no lookup of its own (the walks read the segment bounds from
    // global memory).
    bool ok = true;
    const int my_steps = idle ? 0 : J;
    int u = 0, piece_end = 0, cur_kf = 0, nu = 0, nxt_kf = 0, nxt_len = 0;
    bool need_next = false;
    auto look_ahead = [&]() {
      need_next = false;
      nu = next_busy_unit(a, u + 1);
      const Piece q = piece_at(a, nu);
      nxt_kf = q.kind | (q.n_fix << 2);
      nxt_len = q.c_hi - q.c_lo;
    };
    if (my_steps > 0) {
      u = next_busy_unit(a, units_begin(a));
      const Piece q = piece_at(a, u);
      cur_kf = q.kind | (q.n_fix << 2);
      piece_end = q.c_hi - q.c_lo;
      need_next = piece_end < my_steps;
      conv_init_x(tx);
    }
    for (int j = 0; j < my_steps; ++j) {
      do {
        if (!ok) break;
        const int st = j & 1;
        const uint32_t par = (uint32_t)j & 1u;
        if (j > 0 && !(ok = mbar_wait_sleep(&bar_x[half], par ^ 1u, a.err))) break;  // previous update done
        if (!(ok = mbar_wait_sleep(&bar_full[st], ((uint32_t)j >> 1) & 1u, a.err))) break;
        tc_fence_after();
        const float *sR = reinterpret_cast<const float *>(sm + OFF_SC + st * 512);
        const float gamma_C = sR[C];
        // (1) this thread's 64 rows i of X^T: hi pieces to TMEM, lo pieces to the shared A tile,
        // gamma_C X^T back into the accumulator.
#pragma unroll
        for (int cb = 0; cb < 64; cb += 32) {
          float xv[32];
          tmem_ld32(tx + 64 * part + cb, xv);
          float ph[16];
          uint32_t pl[16];
#pragma unroll
          for (int q = 0; q < 16; ++q) {
            uint32_t hi2;
            split2_pair(xv[2 * q], xv[2 * q + 1], hi2, pl[q]);
            ph[q] = __uint_as_float(hi2);
          }
          tmem_st16(txp + (64 * part + cb) / 2, ph);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            *reinterpret_cast<uint4 *>(xlo + sw128_offset((uint32_t)row, (uint32_t)(cb / 8 + k))) =
                make_uint4(pl[4 * k], pl[4 * k + 1], pl[4 * k + 2], pl[4 * k + 3]);
#pragma unroll
          for (int q = 0; q < 32; ++q) xv[q] *= gamma_C;
          tmem_st32(tx + 64 * part + cb, xv);
        }
        tmem_st_wait();
        fence_proxy_async();
        tc_fence_before();
        mbar_arrive(&bar_r1[half]);
        // (the T-only chain, whose units are the long request bodies, looks up at the boundary)
        if constexpr (!T_ONLY)
          if (need_next) look_ahead();
        // (2) R^T = -(P^T - U^T) diag(exp(G_C - G_t)) -> bf16 hi/lo pieces in place: this thread's
        // columns t in [32 part, 32 part + 32) become 16 hi columns then 16 lo columns.
        if (!(ok = mbar_wait_sleep(&bar_p[half], par, a.err))) break;
        tc_fence_after();
        {
          float pv[32];
          tmem_ld32(tp + 32 * part, pv);
          float ph[16], pl[16];
#pragma unroll
          for (int q = 0; q < 16; ++q) {
            const int t = 32 * part + 2 * q;
            uint32_t hi2, lo2;
            split2_pair(-pv[2 * q] * sR[t], -pv[2 * q + 1] * sR[t + 1], hi2, lo2);
            ph[q] = __uint_as_float(hi2);
            pl[q] = __uint_as_float(lo2);
          }
          tmem_st16(tp + 32 * part, ph);
          tmem_st16(tp + 32 * part + 16, pl);
          tmem_st_wait();
        }
        tc_fence_before();
        mbar_arrive(&bar_r2[half]);
      } while (false);
      if (j + 1 != piece_end) continue;
      // ---- end of a piece: the half's last update has landed
      if (ok) ok = mbar_wait_cycles(&bar_x[half], (uint32_t)j & 1u, a.err);
      tc_fence_after();
      Piece p{};
      if constexpr (T_ONLY) {
        p = piece_at(a, u);
      } else {
        p.s = u / a.Hb;
        p.hh = u % a.Hb;
        p.kind = cur_kf & 3;
        p.n_fix = cur_kf >> 2;
      }
      if (p.kind == PIECE_WHOLE) {
        if (ok) conv_write_x(tx, unit_out(a, p, half));
      } else if constexpr (!T_ONLY) {
        if (p.kind == PIECE_TAIL)
          conv_publish(a, tx, ok);
        else  // PIECE_HEAD, always this CTA's last piece
          ok = conv_compose_head(a, p, tx, txp, xlo, sm, &bar_r1[half], &bar_x[half], J, ok);
      }
      if (j + 1 < my_steps) {
        if constexpr (T_ONLY) {
          u = next_busy_unit(a, u + 1);
          const Piece q = piece_at(a, u);
          piece_end += q.c_hi - q.c_lo;
        } else {
          if (need_next) look_ahead();  // the piece's steps ended early (an error): look it up now
          u = nu;
          cur_kf = nxt_kf;
          piece_end += nxt_len;
          need_next = piece_end < my_steps;
        }
        if (ok) conv_init_x(tx);  // the previous piece's X^T has been read out
      }
    }
    if (!ok) abort_flag = 1;
  }
  __syncthreads();
  tc_fence_after();
  if (abort_flag && tid == 0) {
    // Let any copy or MMA still in flight land before the tensor memory is released.
    for (int k = 0; k < 2; ++k)
      for (int i = 0; i < 2; ++i) {
        mbar_wait_cycles(&bar_x[i], (uint32_t)k, nullptr, 100000000LL);
        mbar_wait_cycles(&bar_p[i], (uint32_t)k, nullptr, 100000000LL);
        mbar_wait_cycles(&bar_full[i], (uint32_t)k, nullptr, 100000000LL);
        mbar_wait_cycles(&bar_empty[i], (uint32_t)k, nullptr, 100000000LL);
      }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, TM_COLS);
}

// ------------------------------------------------------------------------------------------------
// Kernel 3 (builds with per-token outputs): per (segment, head) -- the S half again, with outputs.
//
// Within a chunk, with S_p the state at the chunk start, gamma_t = exp(G_t) and Wm the rows of
// effective writes (Wm = U - Wk S_p, the quantity whose scaled form is R), the post-update state
// of token t is S_t = gamma_t S_p + sum_{s<=t} exp(G_t - G_s) k_s Wm_s^T, so
//   o_t^T = q_t^T S_t:   O^T = S_p^T Q^T diag(gamma) + Wm^T M^T,  M_ts = exp(G_t - G_s) q_t.k_s (s <= t).
// This kernel runs the S-half chain of chain_tc_kernel and adds the two output products: the
// inter-chunk one reuses the state pieces the P product reads (A = S_p^T hi and lo, both kept in
// tensor memory here; B = the chunk's Q tile, exact bf16, K-major), the intra-chunk one takes
// Wm^T in bf16 hi + lo pieces (A, tensor memory) and M from the prep kernel's record (B).  The
// outputs of chunk c are read out (scaled by gamma_t, summed) while chunk c + 1's P product runs;
// gamma_t is kept in registers from the chunk's staged scales, taken before the stage is refilled.
// The state chain's products (U, P, the update) and the two output products are issued by two
// threads (warps 8 and 10): one thread issues an MMA only about every 90 cycles, and the output
// products are off the state's serial path.
// T_C comes from chain_tc_kernel, run for the T half only; this kernel writes S_{C|0} and o.
// Two 32-column TMEM loads of this thread's lane, then one wait for both.
__device__ __forceinline__ void tmem_ld32_pair(uint32_t ta, uint32_t tb, float (&a)[32], float (&b)[32]) {
  uint32_t r[32], u[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%64];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%65];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
        "=r"(u[0]), "=r"(u[1]), "=r"(u[2]), "=r"(u[3]), "=r"(u[4]), "=r"(u[5]), "=r"(u[6]), "=r"(u[7]), "=r"(u[8]), "=r"(u[9]), "=r"(u[10]), "=r"(u[11]), "=r"(u[12]), "=r"(u[13]), "=r"(u[14]), "=r"(u[15]), "=r"(u[16]), "=r"(u[17]), "=r"(u[18]), "=r"(u[19]), "=r"(u[20]), "=r"(u[21]), "=r"(u[22]), "=r"(u[23]), "=r"(u[24]), "=r"(u[25]), "=r"(u[26]), "=r"(u[27]), "=r"(u[28]), "=r"(u[29]), "=r"(u[30]), "=r"(u[31])
      : "r"(ta), "r"(tb)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    a[i] = __uint_as_float(r[i]);
    b[i] = __uint_as_float(u[i]);
  }
}

constexpr uint32_t SO_K = 0, SO_V = 16384, SO_Q = 32768, SO_REC = 49152, SO_M = SO_REC + WS_TILES;
constexpr uint32_t SO_STAGE = SO_M + 16384;  // 112 KB
constexpr uint32_t SO_SMEM = 2 * SO_STAGE + 1024;
constexpr uint32_t SO_X = 0, SO_XH = 128, SO_XL = 192, SO_P = 256, SO_OI = 320, SO_OA = 384, SO_WM = 448;
constexpr int SO_NT = 256 + 96;  // converters + state MMA warp + TMA warp + output MMA warp

__global__ void __launch_bounds__(SO_NT, 1)
    chain_so_kernel(const __grid_constant__ CUtensorMap mapK, const __grid_constant__ CUtensorMap mapV,
                    const __grid_constant__ CUtensorMap mapQ, BuildTcArgs a) {
  extern __shared__ uint8_t smem_raw[];
  // rd: the converters have read chunk c's outputs out (the output accumulators may be reused);
  // oi: the inter-chunk output product has read the state pieces (they may be rewritten)
  __shared__ uint64_t bar_full[2], bar_empty[2], bar_r1, bar_r2, bar_p, bar_x, bar_o, bar_rd, bar_oi;
  __shared__ __align__(16) float s_sc[2][WS_SCG_BYTES / 4];  // scales, gamma_C, gamma_t per stage
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(sm);
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const bool issuer = warp == 8, producer = warp == 9, out_issuer = warp == 10;
  const int row = tid & 127, part = (tid >> 7) & 1;
  const int hh = blockIdx.x % a.Hb;
  const int s = blockIdx.x / a.Hb;
  const int h = a.h0 + hh;
  int64_t beg, end;
  if (!seg_bounds(a, s, beg, end)) return;  // reported by chain_tc_kernel
  const int nchunks = (int)((end - beg + C - 1) / C);

  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar_full[i], 1);
      mbar_init(&bar_empty[i], 2);  // both MMA threads read the stage
    }
    mbar_init(&bar_r1, 256);
    mbar_init(&bar_r2, 256);
    mbar_init(&bar_p, 1);
    mbar_init(&bar_x, 1);
    mbar_init(&bar_o, 1);
    mbar_init(&bar_rd, 256);
    mbar_init(&bar_oi, 1);
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
  const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;

  if (producer) {
    if (lane == 0) {
      prefetch_tmap(&mapK);
      prefetch_tmap(&mapV);
      prefetch_tmap(&mapQ);
      bool ok = true;
      for (int c = 0; c < nchunks && ok; ++c) {
        const int st = c & 1;
        if (c >= 2 && !(ok = mbar_wait_cycles(&bar_empty[st], (uint32_t)((c >> 1) - 1) & 1u, a.err))) break;
        const int rowt = (int)(beg + (int64_t)c * C);
        uint8_t *stg = sm + st * SO_STAGE;
        const uint8_t *rec = ws_rec(a, s, c, hh);
        mbar_arrive_expect_tx(&bar_full[st], 3u * 16384u + WS_TILES + 16384u + WS_SCG_BYTES);
        tma_load_2d(stg + SO_K, &mapK, &bar_full[st], h * D, rowt);
        tma_load_2d(stg + SO_K + 8192, &mapK, &bar_full[st], h * D + 64, rowt);
        tma_load_2d(stg + SO_V, &mapV, &bar_full[st], h * D, rowt);
        tma_load_2d(stg + SO_V + 8192, &mapV, &bar_full[st], h * D + 64, rowt);
        tma_load_2d(stg + SO_Q, &mapQ, &bar_full[st], h * D, rowt);
        tma_load_2d(stg + SO_Q + 8192, &mapQ, &bar_full[st], h * D + 64, rowt);
        bulk_load(stg + SO_REC, rec, WS_TILES, &bar_full[st]);
        bulk_load(stg + SO_M, rec + WS_MH, 16384, &bar_full[st]);
        bulk_load(&s_sc[st][0], rec + WS_SC, WS_SCG_BYTES, &bar_full[st]);
      }
      if (!ok) abort_flag = 1;
    }
    __syncwarp();
  } else if (issuer) {
    if (lane == 0) {
      const uint32_t id_u = idesc_f32acc(1, 1, 1, 0, 128, 64);   // A = V^T (MN-major), B K-major
      const uint32_t id_p = idesc_f32acc(1, 1, 0, 1, 128, 64);   // A = X^T pieces, B = Wk^T (MN-major)
      const uint32_t id_x = idesc_f32acc(1, 1, 0, 1, 128, 128);  // A = R^T pieces, B = K (MN-major)
      auto stage_ready = [&](int c) -> bool {
        const uint32_t stg = sb + (c & 1) * SO_STAGE;
        if (!mbar_wait_cycles(&bar_full[c & 1], ((uint32_t)c >> 1) & 1u, a.err)) return false;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t av = sdesc_sw128(stg + SO_V + kk * 2048, 8192, 1024);
          mma_f16(tmem + SO_P, av, sdesc_sw128(stg + SO_REC + WS_AVH + kk * 32, 16, 1024), id_u, kk > 0);
          mma_f16(tmem + SO_P, av, sdesc_sw128(stg + SO_REC + WS_AVL + kk * 32, 16, 1024), id_u, 1);
        }
        return true;
      };
      bool ok = nchunks == 0 || stage_ready(0);
      for (int c = 0; c < nchunks && ok; ++c) {
        const uint32_t par = (uint32_t)c & 1u;
        const uint32_t stg = sb + (c & 1) * SO_STAGE;
        if (!(ok = mbar_wait_cycles(&bar_r1, par, a.err))) break;
        tc_fence_after();
        // P^T += X^T Wk^T (hi.hi + hi.lo + lo.hi)
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t wh = sdesc_sw128(stg + SO_REC + WS_WH + kk * 2048, 16384, 1024);
          const uint64_t wl = sdesc_sw128(stg + SO_REC + WS_WL + kk * 2048, 16384, 1024);
          mma_f16_tmem_a(tmem + SO_P, tmem + SO_XH + kk * 8, wh, id_p, 1);
          mma_f16_tmem_a(tmem + SO_P, tmem + SO_XH + kk * 8, wl, id_p, 1);
          mma_f16_tmem_a(tmem + SO_P, tmem + SO_XL + kk * 8, wh, id_p, 1);
        }
        mma_commit(&bar_p);
        if (!(ok = mbar_wait_cycles(&bar_r2, par, a.err))) break;
        tc_fence_after();
        // X^T += R^T K
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t bk = sdesc_sw128(stg + SO_K + kk * 2048, 8192, 1024);
          const uint32_t pc = tmem + SO_P + 32 * (kk >> 1) + 8 * (kk & 1);
          mma_f16_tmem_a(tmem + SO_X, pc, bk, id_x, 1);
          mma_f16_tmem_a(tmem + SO_X, pc + 16, bk, id_x, 1);
        }
        mma_commit(&bar_x);
        mma_commit(&bar_empty[c & 1]);
        if (c + 1 < nchunks && !(ok = stage_ready(c + 1))) break;
      }
      if (!ok) abort_flag = 1;
    }
    __syncwarp();
  } else if (out_issuer) {
    // the output products of every chunk, beside the state chain
    if (lane == 0) {
      const uint32_t id_k = idesc_f32acc(1, 1, 0, 0, 128, 64);  // A = TMEM pieces, B K-major (Q, M)
      bool ok = true;
      for (int c = 0; c < nchunks && ok; ++c) {
        const uint32_t par = (uint32_t)c & 1u;
        const uint32_t stg = sb + (c & 1) * SO_STAGE;
        // the chunk's state pieces are written (and its stage landed, which r1 follows)
        if (!(ok = mbar_wait_cycles(&bar_r1, par, a.err))) break;
        // the previous chunk's outputs must have been read out before the accumulators are reused
        if (c > 0 && !(ok = mbar_wait_cycles(&bar_rd, par ^ 1u, a.err))) break;
        tc_fence_after();
        // O_inter^T = X^T Q^T (hi + lo; Q exact)
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t bq = sdesc_sw128(stg + SO_Q + (kk >> 2) * 8192 + (kk & 3) * 32, 16, 1024);
          mma_f16_tmem_a(tmem + SO_OI, tmem + SO_XH + kk * 8, bq, id_k, kk > 0);
          mma_f16_tmem_a(tmem + SO_OI, tmem + SO_XL + kk * 8, bq, id_k, 1);
        }
        mma_commit(&bar_oi);
        if (!(ok = mbar_wait_cycles(&bar_r2, par, a.err))) break;
        tc_fence_after();
        // O_intra^T = Wm^T M^T (hi.hi + hi.lo + lo.hi)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t mh = sdesc_sw128(stg + SO_M + kk * 32, 16, 1024);
          const uint64_t ml = sdesc_sw128(stg + SO_M + 8192 + kk * 32, 16, 1024);
          const uint32_t wc = tmem + SO_WM + 32 * (kk >> 1) + 8 * (kk & 1);
          mma_f16_tmem_a(tmem + SO_OA, wc, mh, id_k, kk > 0);
          mma_f16_tmem_a(tmem + SO_OA, wc, ml, id_k, 1);
          mma_f16_tmem_a(tmem + SO_OA, wc + 16, mh, id_k, 1);
        }
        mma_commit(&bar_o);
        mma_commit(&bar_empty[c & 1]);
      }
      if (!ok) abort_flag = 1;
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ conversion warps (0-7)
    const uint32_t tx = tmem + lane_base + SO_X, tp = tmem + lane_base + SO_P;
    for (int c0 = 64 * part; c0 < 64 * part + 64; c0 += 16) {
      float v[16];
#pragma unroll
      for (int q = 0; q < 16; ++q) v[q] = 0.f;
      tmem_st16(tx + c0, v);
    }
    tmem_st_wait();
    // Outputs of chunk cc: o_t[j] = gamma_t O_inter[j][t] + O_intra[j][t], this thread's 32 t, with
    // gamma_t taken from the staged scales while the chunk's stage still held them.
    float gam[32];
    auto readout = [&](int cc) {
      float oi[32], oa[32];
      tmem_ld32_pair(tmem + lane_base + SO_OI + 32 * part, tmem + lane_base + SO_OA + 32 * part, oi, oa);
      const int64_t t0 = beg + (int64_t)cc * C;
#pragma unroll
      for (int q = 0; q < 32; ++q) {
        const int t = 32 * part + q;
        if (t0 + t < end) a.o_out[((size_t)(t0 + t) * a.H + h) * D + row] = fmaf(gam[q], oi[q], oa[q]);
      }
    };
    bool ok = true;
    for (int c = 0; c < nchunks && ok; ++c) {
      const int st = c & 1;
      const uint32_t par = (uint32_t)c & 1u;
      if (c > 0 && !(ok = mbar_wait_cycles(&bar_x, par ^ 1u, a.err))) break;  // previous update done
      // and the previous chunk's inter-chunk output product has read the state pieces
      if (c > 0 && !(ok = mbar_wait_cycles(&bar_oi, par ^ 1u, a.err))) break;
      if (!(ok = mbar_wait_cycles(&bar_full[st], ((uint32_t)c >> 1) & 1u, a.err))) break;
      tc_fence_after();
      const float *sR = s_sc[st];
      const float gamma_C = sR[C];
      // (1) X^T (= S_p^T) -> hi and lo pieces in tensor memory; gamma_C X^T back.
#pragma unroll
      for (int cb = 0; cb < 64; cb += 32) {
        float xv[32];
        tmem_ld32(tx + 64 * part + cb, xv);
        float ph[16], pl[16];
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          uint32_t hi, lo;
          split2_pair(xv[2 * q], xv[2 * q + 1], hi, lo);
          ph[q] = __uint_as_float(hi);
          pl[q] = __uint_as_float(lo);
        }
        tmem_st16(tmem + lane_base + SO_XH + (64 * part + cb) / 2, ph);
        tmem_st16(tmem + lane_base + SO_XL + (64 * part + cb) / 2, pl);
#pragma unroll
        for (int q = 0; q < 32; ++q) xv[q] *= gamma_C;
        tmem_st32(tx + 64 * part + cb, xv);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bar_r1);
      if (c > 0) {
        // chunk c - 1's outputs, while this chunk's P product runs
        if (!(ok = mbar_wait_cycles(&bar_o, par ^ 1u, a.err))) break;
        tc_fence_after();
        readout(c - 1);
        tc_fence_before();
        mbar_arrive(&bar_rd);
      }
      // this chunk's gamma_t for its readout in the next step (the stage is refilled only after
      // this chunk's last products)
#pragma unroll
      for (int q = 0; q < 32; ++q) gam[q] = sR[(WS_GAM - WS_SC) / 4 + 32 * part + q];
      // (2) Wm^T = -(P^T - U^T): R^T = Wm^T diag(exp(G_C - G_t)) pieces in place, Wm^T pieces aside.
      if (!(ok = mbar_wait_cycles(&bar_p, par, a.err))) break;
      tc_fence_after();
      {
        float pv[32];
        tmem_ld32(tp + 32 * part, pv);
        float rh[16], rl[16], wh[16], wl[16];
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          const int t = 32 * part + 2 * q;
          uint32_t hi, lo;
          split2_pair(-pv[2 * q] * sR[t], -pv[2 * q + 1] * sR[t + 1], hi, lo);
          rh[q] = __uint_as_float(hi);
          rl[q] = __uint_as_float(lo);
          split2_pair(-pv[2 * q], -pv[2 * q + 1], hi, lo);
          wh[q] = __uint_as_float(hi);
          wl[q] = __uint_as_float(lo);
        }
        tmem_st16(tp + 32 * part, rh);
        tmem_st16(tp + 32 * part + 16, rl);
        tmem_st16(tmem + lane_base + SO_WM + 32 * part, wh);
        tmem_st16(tmem + lane_base + SO_WM + 32 * part + 16, wl);
        tmem_st_wait();
      }
      tc_fence_before();
      mbar_arrive(&bar_r2);
    }
    if (ok && nchunks > 0) {
      if ((ok = mbar_wait_cycles(&bar_o, (uint32_t)(nchunks - 1) & 1u, a.err))) {
        tc_fence_after();
        readout(nchunks - 1);
      }
    }
    // the last update has landed: its commit is the state MMA thread's, which the output products'
    // commit does not order
    if (ok && nchunks > 0) {
      ok = mbar_wait_cycles(&bar_x, (uint32_t)(nchunks - 1) & 1u, a.err);
      tc_fence_after();
    }
    if (ok) {
      // S_{C|0}: X^T lane j holds column j; this thread's 64 rows i.
      float *out = a.S_out + ((size_t)s * a.H + h) * D * D;
#pragma unroll
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
  if (abort_flag && tid == 0) {
    for (int k = 0; k < 2; ++k) {
      mbar_wait_cycles(&bar_o, (uint32_t)k, nullptr, 100000000LL);
      mbar_wait_cycles(&bar_oi, (uint32_t)k, nullptr, 100000000LL);
      mbar_wait_cycles(&bar_rd, (uint32_t)k, nullptr, 100000000LL);
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

size_t bytes_per_head(int n_seg, int64_t max_len, bool want_o) {
  const int64_t chunks = (max_len + C - 1) / C;
  return (size_t)n_seg * (size_t)(chunks > 0 ? chunks : 1) * (want_o ? WS_REC_O : WS_REC);
}

// Pair slots of the split chain schedule, after the records: one (T, S) pair per chain CTA (at
// most kSplitSlots CTAs), then a publish flag each and the CTAs' schedule (two ints each).  With
// fewer units than SMs a unit may be cut several times, into pieces of at least kMinPiece chunk
// steps, so the slots are counted from the chunk steps as well.
constexpr int kSplitSlots = 256;
constexpr int kMinPiece = 8;
constexpr size_t kSlotBytes = 2 * D * D * sizeof(float);
int split_slots(long long units, long long steps) {
  long long n = steps / kMinPiece > units ? steps / kMinPiece : units;
  return (int)(n < kSplitSlots ? (n > 0 ? n : 0) : kSplitSlots);
}
size_t split_bytes(long long units, long long steps) {
  const int n = split_slots(units, steps);
  return n ? (size_t)n * kSlotBytes + 3 * kSplitSlots * sizeof(int) : 0;  // + flags and schedule
}

// Chain CTAs the device keeps resident at once in a cooperative launch (0: no cooperative launch).
int chain_resident_ctas() {
  static int cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (cache[dev] == 0) {
    int sms = 0, coop = 0, per = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, chain_tc_kernel<false>, NT2, SMEM_BYTES) != cudaSuccess)
      return 0;
    cache[dev] = (coop && sms * per > 0) ? sms * per : -1;
  }
  return cache[dev] > 0 ? cache[dev] : 0;
}

}  // namespace

bool build_tc_supported(int D_, int fam, int in_dtype, bool want_o) {
  (void)want_o;  // with or without per-token outputs
  return D_ == D && in_dtype == HYPIC_BF16 && (fam == HYPIC_FAM_DELTA || fam == HYPIC_FAM_GATED_DELTA);
}

size_t build_tc_min_workspace(int n_seg, int64_t max_len, bool want_o) {
  return bytes_per_head(n_seg, max_len, want_o);
}

size_t build_tc_workspace_bytes(int H, int n_seg, int64_t max_len, bool want_o) {
  if (H <= 0 || n_seg <= 0) return 0;
  const size_t per = bytes_per_head(n_seg, max_len, want_o);
  size_t heads = WS_CAP / per;
  if (heads < 1) heads = 1;
  if (heads > (size_t)H) heads = (size_t)H;
  const long long units = (long long)n_seg * (long long)heads;
  const int64_t chunks = (max_len + C - 1) / C;
  return heads * per + (want_o ? 0 : split_bytes(units, units * (chunks > 0 ? chunks : 1)));
}

// Runs the build over head blocks that fit the workspace: prep then chain for each block (and,
// with per-token outputs, the S chain that emits them).
// The outputs build runs its two chains (T half; S half with outputs) side by side: both read the
// same records and write disjoint outputs, so the T-half chain goes to a side stream forked after
// the prep kernel and joined back before the next head block's prep.  One side stream and two
// events per device, created on first use; the enqueue holds a per-device lock so that calls from
// several host threads do not interleave their fork and join.
struct SideStream {
  cudaStream_t s = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};
constexpr int kMaxSideDevices = 64;
bool side_stream(int dev, SideStream **out, std::mutex **mu_out) {
  static std::mutex mu[kMaxSideDevices];
  static SideStream side[kMaxSideDevices];
  static bool ready[kMaxSideDevices];
  if (dev < 0 || dev >= kMaxSideDevices) return false;
  std::lock_guard<std::mutex> g(mu[dev]);
  if (!ready[dev]) {
    if (cudaStreamCreateWithFlags(&side[dev].s, cudaStreamNonBlocking) != cudaSuccess) return false;
    if (cudaEventCreateWithFlags(&side[dev].fork, cudaEventDisableTiming) != cudaSuccess) return false;
    if (cudaEventCreateWithFlags(&side[dev].join, cudaEventDisableTiming) != cudaSuccess) return false;
    ready[dev] = true;
  }
  *out = &side[dev];
  *mu_out = &mu[dev];
  return true;
}

cudaError_t launch_build_tc(const RecurrentArgs &r, void *ws, size_t ws_bytes, cudaStream_t st) {
  const bool wo = r.o_out != nullptr;
  const size_t per = bytes_per_head(r.n_seg, r.seg.max_len, wo);
  const int hb_max = (int)((ws_bytes / per) < (size_t)r.H ? ws_bytes / per : (size_t)r.H);
  if (hb_max < 1 || ws == nullptr) return cudaErrorMemoryAllocation;
  // as few blocks as the workspace allows, of equal size (no small tail block)
  const int nblk = (r.H + hb_max - 1) / hb_max;
  const int Hb = (r.H + nblk - 1) / nblk;
  BuildTcArgs a{};
  a.H = r.H;
  a.n_seg = r.n_seg;
  a.bounds = r.seg.bounds;
  a.len0 = r.seg.bounds ? 0 : r.seg.uni_len;
  a.max_len = r.seg.max_len;
  a.n_tokens = r.seg.n_tokens < 0 ? INT64_MAX : r.seg.n_tokens;
  a.max_chunks = (int)((r.seg.max_len + C - 1) / C);
  if (a.max_chunks < 1) a.max_chunks = 1;
  a.fam = r.fam;
  a.alpha = r.src.alpha;
  a.beta = r.src.beta;
  a.T_out = r.T_out;
  a.S_out = r.S_out;
  a.o_out = r.o_out;
  a.ws = static_cast<uint8_t *>(ws);
  a.rec_bytes = wo ? WS_REC_O : WS_REC;
  a.err = r.err;
  const uint64_t n_tok = r.seg.n_tokens < 0 ? (uint64_t)1 << 31 : (uint64_t)r.seg.n_tokens;
  CUtensorMap mk, mv, mq;
  if (!make_tmap_bf16_2d(&mk, r.src.k, n_tok, (uint64_t)r.H * D, (uint64_t)r.H * D, 64, 64))
    return cudaErrorInvalidValue;
  if (!make_tmap_bf16_2d(&mv, r.src.v, n_tok, (uint64_t)r.H * D, (uint64_t)r.H * D, 64, 64))
    return cudaErrorInvalidValue;
  if (wo) {
    if (!make_tmap_bf16_2d(&mq, r.src.q, n_tok, (uint64_t)r.H * D, (uint64_t)r.H * D, 64, 64))
      return cudaErrorInvalidValue;
  } else {
    mq = mk;  // not read
  }
  cudaError_t e = wo ? cudaFuncSetAttribute(wy_prep_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, P_SMEM_O)
                     : cudaFuncSetAttribute(wy_prep_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, P_SMEM);
  if (e != cudaSuccess) return e;
  e = wo ? cudaFuncSetAttribute(chain_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES)
         : cudaFuncSetAttribute(chain_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) return e;
  if (wo) {
    e = cudaFuncSetAttribute(chain_so_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SO_SMEM);
    if (e != cudaSuccess) return e;
  }
  SideStream *side = nullptr;
  std::mutex *side_mu = nullptr;
  std::unique_lock<std::mutex> side_lock;
  if (wo) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || !side_stream(dev, &side, &side_mu)) return cudaErrorInvalidResourceHandle;
    side_lock = std::unique_lock<std::mutex>(*side_mu);
  }
  // The split chain schedule needs its pair slots after the records and a cooperative launch.
  const size_t rec_end = (size_t)Hb * per;  // a multiple of 256 bytes
  const bool split_room =
      !wo && ws_bytes >= rec_end + split_bytes((long long)r.n_seg * Hb, (long long)r.n_seg * Hb * a.max_chunks);
  const int resident = split_room ? chain_resident_ctas() : 0;
  for (int h0 = 0; h0 < r.H; h0 += Hb) {
    a.h0 = h0;
    a.Hb = (r.H - h0) < Hb ? (r.H - h0) : Hb;
    const long long g1 = (long long)r.n_seg * a.max_chunks * a.Hb;
    const long long units = (long long)r.n_seg * a.Hb;
    if (g1 > 0x7fffffffLL || units > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    a.n_units = (int)units;
    a.q_steps = a.max_chunks;
    a.part = nullptr;
    a.flags = nullptr;
    a.sched = nullptr;
    a.n_flags = 0;
    long long g2 = units;
    const long long steps = units * a.max_chunks;
    const int slots = split_slots(units, steps);
    const int cap = resident < slots ? resident : slots;
    // More units than resident CTAs: cap CTAs over equal shares of the chunk steps, each unit cut
    // at most once.  Fewer: the same when it shortens the longest share by a quarter or more, the
    // units then cut into pieces of at least kMinPiece steps.
    long long q = 0;
    if (cap > 0 && units > cap) {
      q = (steps + cap - 1) / cap;
    } else if (cap > 0) {
      const long long qm = (steps + cap - 1) / cap;
      q = qm > kMinPiece ? qm : kMinPiece;
      if (4 * q > 3 * (long long)a.max_chunks) q = 0;
    }
    if (q > 0) {
      if (q > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
      a.q_steps = (int)q;
      g2 = (steps + q - 1) / q;
      a.part = reinterpret_cast<float *>(a.ws + rec_end);
      a.flags = reinterpret_cast<int *>(a.ws + rec_end + (size_t)slots * kSlotBytes);
      a.sched = a.flags + kSplitSlots;
      a.n_flags = (int)g2;
    }
    if (wo) wy_prep_kernel<true><<<(unsigned)g1, NT, P_SMEM_O, st>>>(mk, mq, a);
    else wy_prep_kernel<false><<<(unsigned)g1, NT, P_SMEM, st>>>(mk, mq, a);
    if (wo) {
      if ((e = cudaEventRecord(side->fork, st)) != cudaSuccess) return e;
      if ((e = cudaStreamWaitEvent(side->s, side->fork, 0)) != cudaSuccess) return e;
      chain_tc_kernel<true><<<(unsigned)g2, NT2, SMEM_BYTES, side->s>>>(mk, mv, a);
      if ((e = cudaGetLastError()) != cudaSuccess) return e;
      if ((e = cudaEventRecord(side->join, side->s)) != cudaSuccess) return e;
      chain_so_kernel<<<(unsigned)g2, SO_NT, SO_SMEM, st>>>(mk, mv, mq, a);
      if ((e = cudaGetLastError()) != cudaSuccess) return e;
      if ((e = cudaStreamWaitEvent(st, side->join, 0)) != cudaSuccess) return e;
    } else if (a.flags) {
      // CTAs wait on their neighbours: all must be resident together
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3((unsigned)g2);
      cfg.blockDim = dim3(NT2);
      cfg.dynamicSmemBytes = SMEM_BYTES;
      cfg.stream = st;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeCooperative;
      attr[0].val.cooperative = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      e = cudaLaunchKernelEx(&cfg, chain_tc_kernel<false>, mk, mv, a);
      if (e != cudaSuccess) return e;
    } else {
      chain_tc_kernel<false><<<(unsigned)g2, NT2, SMEM_BYTES, st>>>(mk, mv, a);
    }
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace hypic
