// Tensor-core segment build for the scalar and diagonal decay families at d = 128, bf16 inputs.
//
// For T_t = a_t I (a constant or per-token scalar gate) and T_t = diag(alpha_t), with
// u_t = k_t v_t^T (HYPIC, Method, Table 1: "scalar decay" and "diagonal decay" rows), the
// segment pair of the Method's transition-cache definition has a closed form:
//   T_C = prod_t alpha_t,   S_{C|0} = sum_t diag(f_t) k_t v_t^T = Khat^T V,
//   f_t = prod_{s>t} alpha_s  (per key channel; one scalar for the scalar families),
// so the build is one accumulating GEMM over the segment's tokens with the decay folded
// into the K operand.  A unit is one (segment, head); its 64-token chunks are processed from
// the last to the first while the product of the gates already passed is carried, so every
// factor is known when its chunk is processed and the accumulator is never rescaled.
//
// The kernel is persistent (one CTA per SM, units dealt round-robin) and warp-specialised,
// so the chunk stream through shared memory never stops at a unit boundary:
//   warp 8  (producer)  TMA: K, V (and the diagonal family's gates) into NS stages;
//   warps 0-3 (convert) diagonal: suffix factors in fp32 (one thread per key channel scans down
//                       the chunk in place over the gate tile), then Khat = f * k split into
//                       bf16 hi (over K) + lo (over the gate tile); T_C at the end of each unit.
//                       Scalar: Khat^T = (f * k)^T split hi + lo into tensor memory, with the
//                       factors from warp 10;
//   warp 10 (scalar)    the chunk's suffix factors (a warp scan over the gates), one chunk ahead
//                       of the converters (double buffered), and T_C at the end of each unit;
//   warp 9  (MMA)       S += Khat_hi^T V + Khat_lo^T V (M = N = 128, K = 64 per chunk) into
//                       one of two TMEM accumulators, alternating per unit;
//   warps 4-7 (store)   accumulator -> registers -> padded shared rows -> whole-line stores,
//                       overlapping the next unit's chunks.
// Tokens past a segment's end in its last chunk (the first processed) get f = 0 and a gate
// of 1.  Each input byte is read once and each pair written once.  Every wait is bounded; a
// wait that runs out records HYPIC_ETIMEOUT and all roles stop at their next wait.
#include <cuda_bf16.h>
#include <string.h>

#include <mutex>

#include "common.cuh"
#include "tc_ptx.cuh"
#include "tma_host.h"

namespace hypic {
namespace {

using namespace tc;

constexpr int C = 64;
constexpr int D = 128;
constexpr uint32_t BAR_CONV = 1, BAR_EPI = 2;

// Stage layout (1024-aligned): K / Khat hi [2 boxes of 64 t x 64 i, SW128] at 0, V at 16384,
// gates [64 t][128 i] fp32 (diagonal) at 32768, whose first 16 KB later take Khat lo.  The scalar
// families keep Khat (hi and lo) in tensor memory instead, as the MMA's A operand, so their stage
// is the 32 KB of K and V and six stages fit.  After the stages: the store's row buffer.
template <bool DIAG>
struct Cfg {
  static constexpr int NT = DIAG ? 320 : 352;  // the scalar families add the factor warp
  static constexpr uint32_t STAGE = DIAG ? 65536u : 32768u;
  static constexpr int NS = DIAG ? 3 : 6;
  static constexpr uint32_t TX = DIAG ? 65536u : 32768u;
  static constexpr uint32_t OFF_OUT = STAGE * NS;
  static constexpr uint32_t SMEM = OFF_OUT + 128 * 144 + 1024;
};
constexpr uint32_t OFF_V = 16384, OFF_G = 32768;
constexpr uint32_t OUT_STRIDE = 144;  // one padded row of a 32-column block of S, in bytes
// Tensor memory: two accumulators (columns 0 and 128); scalar families: KB buffers of Khat^T pieces
// (lanes = key channels, 32 columns of token pairs each for hi, then lo) from column 256.
constexpr int KB = 3;
constexpr uint32_t TM_KH = 256;

struct DecayArgs {
  int H, n_seg;
  const int64_t *bounds;
  int64_t stride0, offset0, len0;  // without bounds: segment s is [s stride0 + offset0, + len0)
  int64_t max_len, n_tokens;
  int fam;
  const float *alpha;
  float *T_out, *S_out;
  int *err;
};

// Body of unit u: its (segment, head), token range and chunk count; ok = false for a
// malformed range (recorded once, by the converter, and then skipped by every role).
struct Unit {
  int s, h, nch;
  int64_t beg, end;
  bool ok;
};
__device__ __forceinline__ Unit unit_of(const DecayArgs &a, int u) {
  Unit r;
  r.s = u / a.H;
  r.h = u % a.H;
  if (a.bounds) {
    r.beg = a.bounds[2 * r.s];
    r.end = a.bounds[2 * r.s + 1];
  } else {
    r.beg = (int64_t)r.s * a.stride0 + a.offset0;
    r.end = r.beg + a.len0;
  }
  r.ok = r.beg >= 0 && r.end >= r.beg && r.end - r.beg <= a.max_len && r.end <= a.n_tokens;
  r.nch = r.ok ? (int)((r.end - r.beg + C - 1) / C) : 0;
  return r;
}

// Bounded wait that also gives up as soon as another role has given up.
__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, uint32_t parity, volatile int *abort, int *err) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (*abort) return false;
    if (clock64() - t0 > 2000000000LL) {
      set_error(err, HYPIC_ETIMEOUT);
      *abort = 1;
      return false;
    }
  }
  return true;
}

template <bool DIAG>
__global__ void __launch_bounds__(Cfg<DIAG>::NT, 1)
    build_decay_tc_kernel(const __grid_constant__ CUtensorMap mapK, const __grid_constant__ CUtensorMap mapV,
                          const __grid_constant__ CUtensorMap mapA, DecayArgs a) {
  using G = Cfg<DIAG>;
  constexpr int NS = G::NS;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar_full[NS], bar_conv[NS], bar_empty[NS], bar_acc_full[2], bar_acc_empty[2];
  __shared__ uint64_t bar_kfree[KB];  // scalar families: the MMAs have read a Khat buffer
  __shared__ uint64_t bar_fac_full[2], bar_fac_empty[2];  // scalar families: factors written / read
  __shared__ uint32_t tmem_slot;
  __shared__ volatile int abort_flag;
  __shared__ float s_f[2][C];  // scalar families: factors of the current chunk (double buffered)
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(sm);
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int n_units = a.n_seg * a.H;

  if (tid == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(&bar_full[i], 1);
      mbar_init(&bar_conv[i], 128);
      mbar_init(&bar_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar_acc_full[i], 1);
      mbar_init(&bar_acc_empty[i], 128);
    }
    for (int i = 0; i < KB; ++i) mbar_init(&bar_kfree[i], 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar_fac_full[i], 32);
      mbar_init(&bar_fac_empty[i], 128);
    }
    mbar_fence_init();
    abort_flag = 0;
  }
  constexpr uint32_t TM_ALLOC = DIAG ? 256 : 512;
  if (warp == 0) {
    tmem_alloc(&tmem_slot, TM_ALLOC);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;

  // Producer / MMA bookkeeping for the drain after an abort.
  int n_load[NS];
#pragma unroll
  for (int i = 0; i < NS; ++i) n_load[i] = 0;
  int last_commit = -1;

  if (warp == 8) {
    // ---------------- producer ----------------
    if (lane == 0) {
      prefetch_tmap(&mapK);
      prefetch_tmap(&mapV);
      if (DIAG) prefetch_tmap(&mapA);
      int j = 0;
      bool stop = false;
      for (int u = blockIdx.x; u < n_units && !stop; u += gridDim.x) {
        const Unit U = unit_of(a, u);
        for (int q = 0; q < U.nch; ++q, ++j) {
          const int st = j % NS;
          if (j >= NS && !wait_or_abort(&bar_empty[st], (uint32_t)((j / NS - 1) & 1), &abort_flag, a.err)) {
            stop = true;
            break;
          }
          const int row = (int)(U.beg + (int64_t)(U.nch - 1 - q) * C);
          uint8_t *base = sm + st * G::STAGE;
          mbar_arrive_expect_tx(&bar_full[st], G::TX);
          tma_load_2d(base, &mapK, &bar_full[st], U.h * D, row);
          tma_load_2d(base + 8192, &mapK, &bar_full[st], U.h * D + 64, row);
          tma_load_2d(base + OFF_V, &mapV, &bar_full[st], U.h * D, row);
          tma_load_2d(base + OFF_V + 8192, &mapV, &bar_full[st], U.h * D + 64, row);
          if (DIAG) tma_load_2d(base + OFF_G, &mapA, &bar_full[st], U.h * D, row);
          ++n_load[st];
        }
      }
    }
    __syncwarp();
  } else if (warp == 9) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      // A = Khat^T (MN-major in shared memory, or from tensor memory for the scalar families), B = V
      const uint32_t idesc = DIAG ? idesc_f32acc(1, 1, 1, 1, 128, 128) : idesc_f32acc(1, 1, 0, 1, 128, 128);
      int j = 0, m = 0;
      bool stop = false;
      for (int u = blockIdx.x; u < n_units && !stop; u += gridDim.x) {
        const Unit U = unit_of(a, u);
        if (U.nch == 0) continue;
        const int acc = m & 1;
        if (m >= 2 && !wait_or_abort(&bar_acc_empty[acc], (uint32_t)((m / 2 - 1) & 1), &abort_flag, a.err)) break;
        for (int q = 0; q < U.nch; ++q, ++j) {
          const int st = j % NS;
          if (!wait_or_abort(&bar_conv[st], (uint32_t)((j / NS) & 1), &abort_flag, a.err)) {
            stop = true;
            break;
          }
          tc_fence_after();
          const uint32_t kb = sb + st * G::STAGE;
          const uint32_t kt = tmem + TM_KH + (uint32_t)(j % KB) * 64;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t bv = sdesc_sw128(kb + OFF_V + kk * 2048, 8192, 1024);
            if constexpr (DIAG) {
              mma_f16(tmem + acc * 128, sdesc_sw128(kb + kk * 2048, 8192, 1024), bv, idesc, (q | kk) != 0);
              mma_f16(tmem + acc * 128, sdesc_sw128(kb + OFF_G + kk * 2048, 8192, 1024), bv, idesc, 1);
            } else {
              mma_f16_tmem_a(tmem + acc * 128, kt + kk * 8, bv, idesc, (q | kk) != 0);
              mma_f16_tmem_a(tmem + acc * 128, kt + 32 + kk * 8, bv, idesc, 1);
            }
          }
          mma_commit(&bar_empty[st]);
          if constexpr (!DIAG) mma_commit(&bar_kfree[j % KB]);
          last_commit = j;
          if (q == U.nch - 1) mma_commit(&bar_acc_full[acc]);
        }
        ++m;
      }
    }
    __syncwarp();
  } else if (!DIAG && warp < 4) {
    // ---------------- scalar converters (tid = key channel) ----------------
    // Khat^T row i = f_t k_ti over the chunk's tokens, hi and lo pieces into tensor memory (lane i,
    // token pairs per column) once the MMAs of chunk j - KB have read the buffer.  No block-wide
    // barrier: every wait is the thread's own, so a role that stops leaves no one at a barrier.
    int j = 0;
    bool stop = false;
    for (int u = blockIdx.x; u < n_units && !stop; u += gridDim.x) {
      const Unit U = unit_of(a, u);
      if (!U.ok) {
        if (tid == 0) set_error(a.err, HYPIC_EDEVICE);
        continue;
      }
      for (int q = 0; q < U.nch; ++q, ++j) {
        const int st = j % NS, fb = j & 1, buf = j % KB;
        const uint8_t *base = sm + st * G::STAGE;
        if (!wait_or_abort(&bar_full[st], (uint32_t)((j / NS) & 1), &abort_flag, a.err) ||
            !wait_or_abort(&bar_fac_full[fb], (uint32_t)((j >> 1) & 1), &abort_flag, a.err) ||
            (j >= KB && !wait_or_abort(&bar_kfree[buf], (uint32_t)((j / KB - 1) & 1), &abort_flag, a.err))) {
          stop = true;
          break;
        }
        tc_fence_after();
        const int i = tid;
        const uint8_t *kcol = base + (uint32_t)(i >> 6) * 8192u + (uint32_t)(i & 7) * 2u;
        const uint32_t ck = (uint32_t)((i & 63) >> 3);
        const float *ft = s_f[fb];
        float hw[32], lw[32];
#pragma unroll
        for (int t = 0; t < C; t += 2) {
          const float k0 = __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(kcol + sw128_offset((uint32_t)t, ck)));
          const float k1 =
              __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(kcol + sw128_offset((uint32_t)t + 1, ck)));
          const float x0 = ft[t] * k0, x1 = ft[t + 1] * k1;
          const __nv_bfloat162 hp = __floats2bfloat162_rn(x0, x1);
          const float2 hf = __bfloat1622float2(hp);
          const __nv_bfloat162 lp = __floats2bfloat162_rn(x0 - hf.x, x1 - hf.y);
          hw[t / 2] = __uint_as_float(*reinterpret_cast<const uint32_t *>(&hp));
          lw[t / 2] = __uint_as_float(*reinterpret_cast<const uint32_t *>(&lp));
        }
        mbar_arrive(&bar_fac_empty[fb]);  // the factors are in registers
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        tmem_st32(tmem + lane_base + TM_KH + (uint32_t)buf * 64, hw);
        tmem_st32(tmem + lane_base + TM_KH + (uint32_t)buf * 64 + 32, lw);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bar_conv[st]);
      }
    }
  } else if (!DIAG && warp == 10) {
    // ---------------- scalar factors, one chunk ahead of the converters ----------------
    // f_t = product of the gates after token t within the segment (0 past its end); lane l owns
    // tokens 2l and 2l + 1 of the chunk.
    int j = 0;
    bool stop = false;
    for (int u = blockIdx.x; u < n_units && !stop; u += gridDim.x) {
      const Unit U = unit_of(a, u);
      if (!U.ok) continue;
      float carry = 1.f;  // product of the gates of the chunks already passed
      const float gc = a.fam == HYPIC_FAM_SCALAR_CONST ? a.alpha[U.h] : 1.f;
      for (int q = 0; q < U.nch; ++q, ++j) {
        const int fb = j & 1;
        if (j >= 2 && !wait_or_abort(&bar_fac_empty[fb], (uint32_t)(((j >> 1) - 1) & 1), &abort_flag, a.err)) {
          stop = true;
          break;
        }
        const int64_t t0 = U.beg + (int64_t)(U.nch - 1 - q) * C;
        const int nvalid = (int)((U.end - t0) < C ? (U.end - t0) : C);
        const int ta = 2 * lane, tb = 2 * lane + 1;
        float g0 = 1.f, g1 = 1.f;
        if (a.fam == HYPIC_FAM_SCALAR_CONST) {
          g0 = ta < nvalid ? gc : 1.f;
          g1 = tb < nvalid ? gc : 1.f;
        } else {
          if (ta < nvalid) g0 = a.alpha[(t0 + ta) * a.H + U.h];
          if (tb < nvalid) g1 = a.alpha[(t0 + tb) * a.H + U.h];
        }
        float suf = g0 * g1;  // inclusive suffix product over lanes >= lane
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float y = __shfl_down_sync(0xffffffffu, suf, o);
          if (lane + o < 32) suf *= y;
        }
        float after = __shfl_down_sync(0xffffffffu, suf, 1);
        if (lane == 31) after = 1.f;
        const float total = __shfl_sync(0xffffffffu, suf, 0);
        s_f[fb][tb] = tb < nvalid ? carry * after : 0.f;
        s_f[fb][ta] = ta < nvalid ? carry * after * g1 : 0.f;
        carry *= total;
        mbar_arrive(&bar_fac_full[fb]);
      }
      if (!stop && lane == 0) a.T_out[(size_t)U.s * a.H + U.h] = carry;
    }
  } else if (warp < 4) {
    // ---------------- diagonal converters (tid = key channel) ----------------
    if constexpr (DIAG) {
      int j = 0;
      for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
        const Unit U = unit_of(a, u);
        if (!U.ok) {
          if (tid == 0) set_error(a.err, HYPIC_EDEVICE);
          continue;
        }
        float carry = 1.f;  // product of the gates passed, channel tid
        bool stop = false;
        for (int q = 0; q < U.nch; ++q, ++j) {
          const int st = j % NS;
          uint8_t *base = sm + st * G::STAGE;
          const int64_t t0 = U.beg + (int64_t)(U.nch - 1 - q) * C;
          const int nvalid = (int)((U.end - t0) < C ? (U.end - t0) : C);
          const bool ok = wait_or_abort(&bar_full[st], (uint32_t)((j / NS) & 1), &abort_flag, a.err);
          if (bar_or_named(BAR_CONV, 128, !ok)) {
            stop = true;
            break;
          }
          // (1) suffix factors, in place over the gate tile
          {
            float *g = reinterpret_cast<float *>(base + OFF_G);
            float acc = carry;
#pragma unroll 8
            for (int t = C - 1; t >= 0; --t) {
              const float gv = g[t * D + tid];
              const bool v = t < nvalid;
              g[t * D + tid] = v ? acc : 0.f;
              acc = v ? acc * gv : acc;
            }
            carry = acc;
          }
          bar_sync_named(BAR_CONV, 128);
          // (2) Khat = f * k: hi over K in place, lo into the lo slot.  The lo slot overlaps the
          // factor tile, so all factors are read before any lo is written.
          uint32_t lo_w[8][4];
#pragma unroll
          for (int r = 0; r < 8; ++r) {
            const int e = tid + r * 128;
            const int t = e >> 4, c8 = e & 15;  // token t, key channels 8 c8 .. 8 c8 + 7
            const uint32_t off = (uint32_t)(c8 >> 3) * 8192 + sw128_offset((uint32_t)t, (uint32_t)(c8 & 7));
            const uint4 kr = *reinterpret_cast<const uint4 *>(base + off);
            const __nv_bfloat162 *k2 = reinterpret_cast<const __nv_bfloat162 *>(&kr);
            const float *fp = reinterpret_cast<const float *>(base + OFF_G) + t * D + 8 * c8;
            const float4 f0 = *reinterpret_cast<const float4 *>(fp);
            const float4 f1 = *reinterpret_cast<const float4 *>(fp + 4);
            const float f[8] = {f0.x, f0.y, f0.z, f0.w, f1.x, f1.y, f1.z, f1.w};
            uint32_t hi[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float2 kv = __bfloat1622float2(k2[i]);
              const float x0 = kv.x * f[2 * i], x1 = kv.y * f[2 * i + 1];
              const __nv_bfloat162 hp = __floats2bfloat162_rn(x0, x1);
              const float2 hf = __bfloat1622float2(hp);
              const __nv_bfloat162 lp = __floats2bfloat162_rn(x0 - hf.x, x1 - hf.y);
              hi[i] = *reinterpret_cast<const uint32_t *>(&hp);
              lo_w[r][i] = *reinterpret_cast<const uint32_t *>(&lp);
            }
            *reinterpret_cast<uint4 *>(base + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
          }
          bar_sync_named(BAR_CONV, 128);
#pragma unroll
          for (int r = 0; r < 8; ++r) {
            const int e = tid + r * 128;
            const int t = e >> 4, c8 = e & 15;
            const uint32_t off = (uint32_t)(c8 >> 3) * 8192 + sw128_offset((uint32_t)t, (uint32_t)(c8 & 7));
            *reinterpret_cast<uint4 *>(base + OFF_G + off) =
                make_uint4(lo_w[r][0], lo_w[r][1], lo_w[r][2], lo_w[r][3]);
          }
          fence_proxy_async();
          mbar_arrive(&bar_conv[st]);
        }
        if (stop) break;
        a.T_out[((size_t)U.s * a.H + U.h) * D + tid] = carry;
      }
    }
  } else {
    // ---------------- store (warps 4-7; row = TMEM lane = et) ----------------
    const int et = tid - 128;
    const uint32_t lane_base = (uint32_t)((warp - 4) * 32) << 16;
    uint8_t *rows = sm + G::OFF_OUT;
    int m = 0;
    for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
      const Unit U = unit_of(a, u);
      if (!U.ok) continue;
      float *out = a.S_out + ((size_t)U.s * a.H + U.h) * D * D;
      if (U.nch == 0) {
        for (int e = et; e < D * D / 4; e += 128)
          reinterpret_cast<float4 *>(out)[e] = make_float4(0.f, 0.f, 0.f, 0.f);
        continue;
      }
      const int acc = m & 1;
      const bool ok = wait_or_abort(&bar_acc_full[acc], (uint32_t)((m / 2) & 1), &abort_flag, a.err);
      if (bar_or_named(BAR_EPI, 128, !ok)) break;
      tc_fence_after();
#pragma unroll 1
      for (int cb = 0; cb < D; cb += 32) {
        float v[32];
        tmem_ld32(tmem + acc * 128 + lane_base + cb, v);
#pragma unroll
        for (int i = 0; i < 8; ++i)
          *reinterpret_cast<float4 *>(rows + et * OUT_STRIDE + i * 16) =
              make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
        bar_sync_named(BAR_EPI, 128);
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          const int e = et + r * 128;
          const int row = e >> 3, c4 = e & 7;
          const float4 x = *reinterpret_cast<const float4 *>(rows + row * OUT_STRIDE + c4 * 16);
          *reinterpret_cast<float4 *>(out + (size_t)row * D + cb + c4 * 4) = x;
        }
        bar_sync_named(BAR_EPI, 128);
      }
      tc_fence_before();
      mbar_arrive(&bar_acc_empty[acc]);
      ++m;
    }
  }

  __syncthreads();
  if (abort_flag) {
    // Let every copy and MMA in flight land before the shared memory and TMEM go away.
    if (warp == 8 && lane == 0)
      for (int i = 0; i < NS; ++i)
        if (n_load[i]) mbar_wait_cycles(&bar_full[i], (uint32_t)((n_load[i] - 1) & 1), nullptr, 100000000LL);
    if (warp == 9 && lane == 0 && last_commit >= 0)
      mbar_wait_cycles(&bar_empty[last_commit % NS], (uint32_t)((last_commit / NS) & 1), nullptr, 100000000LL);
    __syncthreads();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, TM_ALLOC);
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

template <bool DIAG>
cudaError_t launch_one(const CUtensorMap &mk, const CUtensorMap &mv, const CUtensorMap &ma, const DecayArgs &a,
                       long long units, cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(build_decay_tc_kernel<DIAG>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       Cfg<DIAG>::SMEM);
  if (e != cudaSuccess) return e;
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  const unsigned grid = (unsigned)(units < sms ? units : sms);
  build_decay_tc_kernel<DIAG><<<grid, Cfg<DIAG>::NT, Cfg<DIAG>::SMEM, st>>>(mk, mv, ma, a);
  return cudaGetLastError();
}

}  // namespace

bool build_decay_tc_supported(int D_, int fam, int in_dtype, bool want_o) {
  return D_ == D && in_dtype == HYPIC_BF16 && !want_o &&
         (fam == HYPIC_FAM_SCALAR_CONST || fam == HYPIC_FAM_SCALAR || fam == HYPIC_FAM_DIAG);
}

cudaError_t launch_build_decay_tc(const RecurrentArgs &r, cudaStream_t st) {
  DecayArgs a{};
  a.H = r.H;
  a.n_seg = r.n_seg;
  a.bounds = r.seg.bounds;
  a.stride0 = r.seg.uni_stride;
  a.offset0 = r.seg.uni_offset;
  a.len0 = r.seg.uni_len;
  a.max_len = r.seg.max_len;
  a.n_tokens = r.seg.n_tokens < 0 ? INT64_MAX : r.seg.n_tokens;
  a.fam = r.fam;
  a.alpha = r.src.alpha;
  a.T_out = r.T_out;
  a.S_out = r.S_out;
  a.err = r.err;
  const long long units = (long long)r.n_seg * r.H;
  if (units <= 0) return cudaSuccess;
  if (units > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  const uint64_t n_tok = r.seg.n_tokens < 0 ? (uint64_t)1 << 31 : (uint64_t)r.seg.n_tokens;
  CUtensorMap mk, mv, ma;
  if (!make_tmap_bf16_2d(&mk, r.src.k, n_tok, (uint64_t)r.H * D, (uint64_t)r.H * D, 64, 64))
    return cudaErrorInvalidValue;
  if (!make_tmap_bf16_2d(&mv, r.src.v, n_tok, (uint64_t)r.H * D, (uint64_t)r.H * D, 64, 64))
    return cudaErrorInvalidValue;
  if (r.fam == HYPIC_FAM_DIAG) {
    if (!make_tmap_f32_rows(&ma, r.src.alpha, n_tok, (uint64_t)r.H * D, 128, 64)) return cudaErrorInvalidValue;
    return launch_one<true>(mk, mv, ma, a, units, st);
  }
  memcpy(&ma, &mk, sizeof(ma));  // not read on the scalar path
  return launch_one<false>(mk, mv, ma, a, units, st);
}

}  // namespace hypic
