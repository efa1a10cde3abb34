// Tensor-core composition chain for the delta families at d = 128: compose, fused request
// assembly (seam advance + compose) and the affine scan.  Plain composition and the scan (no seam
// windows) are dispatched from here to the pipelined kernels of compose_pipe.cu; this kernel runs
// the assembly, whose seam windows need the whole column state between two steps.
//
// Composition applies the cached pairs in prompt order, S <- T_C S + S_{C|0} (HYPIC reading
// notes, Method 2, paper Eq. (6)); assembly first advances the running state through the w
// seam tokens of each inner segment and emits o_i = q_i^T S_i (Method 5, seam windows).
//
// One CTA of 256 threads per (request, head).  Thread (j, half) owns rows 64 half .. 64 half + 63
// of column j of the running state S.  Each step computes the transposed product on tcgen05,
//   D = S_new^T = S^T T^T     (M = 128 columns j, N = 128 rows i, K = 128),
// with the A operand S^T held in tensor memory (the epilogue writes it there, so S never
// touches shared memory) and the B operand T^T = T row-major, streamed by TMA.  fp32 accuracy
// comes from exact three-way bf16 splits of both operands, x = hi + mid + lo, each piece
// taking the next 8 bits of the 24-bit significand by truncation (bit masks, no conversions),
// and the six products hi.hi + hi.mid + mid.hi + hi.lo + mid.mid + lo.hi.  The products are
// accumulated smallest first, so the fp32 accumulator's rounding is paid against the small
// correction terms and only the final eight hi.hi steps round against the full-size value.
// The epilogue adds S_{C|0} column j (TMA-staged), runs the next segment's seam tokens on the
// column in registers (k . S_j, rank-1 update, q . S_j), and splits the column into the three
// A pieces for the next step.  Grid order is head-major, so the requests that share a head's
// pool entries run together and re-read them from L2.
//
// Pairs stored in bf16 (16-bit cache storage, Method 3 Table 3 sizes): T is then an exact bf16
// B operand, so TMA lands it directly in the swizzled K-major layout the MMA reads (double
// buffered: the next step's T loads while this step runs), only the three products
// hi.T + mid.T + lo.T remain, and S_{C|0} is staged in bf16 and added in fp32.
#include <cuda_bf16.h>

#include <type_traits>

#include "tc_ptx.cuh"
#include "tma_host.h"

namespace hypic {
namespace {

using namespace tc;

constexpr int D = 128;
constexpr int NT = 256;
constexpr int R = 64;  // rows of the column each thread owns
constexpr int SG = 8;  // seam tokens per group (one coalesced load, one shared-memory pass)
constexpr int NL = SG * D / NT;  // each thread's share of one token tensor of a group

// fp32 pairs
constexpr uint32_t OFF_TST = 0;                 // T staging, fp32, 4 boxes [128 i][32 k] swizzled
constexpr uint32_t OFF_TB = 65536;              // 3 pieces x 2 k-blocks x [128 i][64 k] bf16 (K-major B)
constexpr uint32_t OFF_S0 = OFF_TB + 3 * 32768;  // S0 staging, fp32 [128 i][128 j], row-major
constexpr uint32_t SMEM_BYTES = OFF_S0 + 65536 + 1024;
// bf16 pairs
constexpr uint32_t OFF_TB16 = 0;       // 2 buffers x 2 k-blocks x [128 i][64 k] bf16 (K-major B), by TMA
constexpr uint32_t OFF_S016 = 65536;   // S0 staging, bf16 [128 i][128 j], row-major
constexpr uint32_t SMEM_BYTES16 = OFF_S016 + 32768 + 1024;

constexpr uint32_t TM_D = 0;    // accumulator D = S_new^T: lanes j, columns i
constexpr uint32_t TM_A = 128;  // three A pieces of S^T, 64 columns each (two bf16 per column)
constexpr uint32_t TM_DOT = 320;  // seam windows: k_t . S_j and q_t . S_j (16 columns)
constexpr uint32_t TM_C = 336;    // seam windows: three pieces of the update's coefficients (24 columns)
constexpr uint32_t SEAM_BT = 24576;  // seam windows: the dot products' B tile, within the S0 staging
constexpr uint32_t TM_COLS = 512;

struct ComposeTcArgs {
  int H, B, n, w;
  int B_major;  // 0: grid is head-major (b fastest)
  const int32_t *idx;
  int64_t pool_size;
  const float *S_init;
  float *S_out;
  int scan;
  float *T_rec, *S_rec;
  int fam;
  int seam_bf16;
  const void *seam_k, *seam_v, *seam_q;
  const float *seam_alpha, *seam_beta;
  float *o_out;
  int *err;
};

// Exact three-way split of two fp32 values into bf16 pieces packed two per 32-bit word:
// hi keeps the sign, exponent and top 7 stored significand bits (a bf16 value); the remainder
// r = x - hi is exact in fp32 and is split the same way; lo = r - mid is then a bf16 value
// (at most 8 significant bits remain), so x = hi + mid + lo holds exactly.
__device__ __forceinline__ void split3_pair(float a, float b, uint32_t &p0, uint32_t &p1, uint32_t &p2) {
  const uint32_t ua = __float_as_uint(a), ub = __float_as_uint(b);
  const float ha = __uint_as_float(ua & 0xFFFF0000u), hb = __uint_as_float(ub & 0xFFFF0000u);
  const float ra = a - ha, rb = b - hb;
  const uint32_t ura = __float_as_uint(ra), urb = __float_as_uint(rb);
  const float ma = __uint_as_float(ura & 0xFFFF0000u), mb = __uint_as_float(urb & 0xFFFF0000u);
  const uint32_t ula = __float_as_uint(ra - ma), ulb = __float_as_uint(rb - mb);
  p0 = __byte_perm(ua, ub, 0x7632);  // upper halves: a in the low word, b in the high word
  p1 = __byte_perm(ura, urb, 0x7632);
  p2 = __byte_perm(ula, ulb, 0x7632);
}

__device__ __forceinline__ void tmem_st8(uint32_t taddr, const float (&v)[8]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7]))
      : "memory");
}

template <typename Tin>
__device__ __forceinline__ float ld_tok(const void *p, size_t i) {
  return to_f32<Tin>(static_cast<const Tin *>(p)[i]);
}

template <typename Tin, bool PB>
__global__ void __launch_bounds__(NT, 1)
    compose_tc_kernel(const __grid_constant__ CUtensorMap mapT, const __grid_constant__ CUtensorMap mapS,
                      ComposeTcArgs a) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar_t[2], bar_s, bar_m, bar_d, bar_u;  // bar_t[1]: second T buffer (bf16 pairs)
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(sm);
  float *sS0 = reinterpret_cast<float *>(sm + (PB ? OFF_S016 : OFF_S0));
  const int tid = threadIdx.x, warp = tid / 32;
  const int H = a.H;
  int b, h;
  bool isT = false;  // scan: the T half (starts at I, no addend)
  if (a.scan) {
    isT = (blockIdx.x & 1) == 0;
    h = blockIdx.x >> 1;
    b = 0;
  } else if (a.B_major) {
    h = blockIdx.x % H;
    b = blockIdx.x / H;
  } else {
    b = blockIdx.x % a.B;
    h = blockIdx.x / a.B;
  }
  const int j = tid & (D - 1);   // the state column (= TMEM lane) this thread serves
  const int half = tid >> 7;     // which 64 rows of it
  const int i0 = half * R;
  const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
  const bool addend = !isT;

  auto entry = [&](int step) -> int64_t {
    int64_t p = a.idx ? (int64_t)a.idx[(size_t)b * a.n + step] : (int64_t)step;
    if (p < 0 || p >= a.pool_size) {
      set_error(a.err, HYPIC_EDEVICE);
      p = 0;
    }
    return p;
  };
  auto issue_T = [&](int step) {
    const int row = (int)((entry(step) * H + h) * D);
    if (PB) {
      const int buf = step & 1;
      mbar_arrive_expect_tx(&bar_t[buf], 32768);
#pragma unroll
      for (int kb = 0; kb < 2; ++kb)
        tma_load_2d(sm + OFF_TB16 + buf * 32768 + kb * 16384, &mapT, &bar_t[buf], kb * 64, row);
    } else {
      mbar_arrive_expect_tx(&bar_t[0], 65536);
#pragma unroll
      for (int kb = 0; kb < 4; ++kb) tma_load_2d(sm + OFF_TST + kb * 16384, &mapT, &bar_t[0], kb * 32, row);
    }
  };
  auto issue_S = [&](int step) {
    const int row = (int)((entry(step) * H + h) * D);
    mbar_arrive_expect_tx(&bar_s, PB ? 32768 : 65536);
    tma_load_2d(sm + (PB ? OFF_S016 : OFF_S0), &mapS, &bar_s, 0, row);
  };

  if (tid == 0) {
    mbar_init(&bar_t[0], 1);
    mbar_init(&bar_t[1], 1);
    mbar_init(&bar_s, 1);
    mbar_init(&bar_m, 1);
    mbar_init(&bar_d, 1);
    mbar_init(&bar_u, 1);
    mbar_fence_init();
    abort_flag = 0;
    prefetch_tmap(&mapT);
    prefetch_tmap(&mapS);
    if (a.n > 0) {
      issue_T(0);
      if (addend) issue_S(0);
    }
  }
  if (warp == 0) {
    tmem_alloc(&tmem_slot, TM_COLS);
    tmem_relinquish();
  }

  // Initial rows i0 .. i0 + 63 of column j.
  float x[R];
  const size_t base_bh = ((size_t)b * H + h) * D * D;
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int i = i0 + r;
    if (a.scan) x[r] = (isT && i == j) ? 1.f : 0.f;
    else x[r] = a.S_init ? a.S_init[base_bh + (size_t)i * D + j] : 0.f;
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;

  // A pieces of S^T: lane j, rows i0.. as 32 columns (two rows per column) of each piece.
  auto write_pieces = [&]() {
#pragma unroll
    for (int c0 = 0; c0 < R; c0 += 16) {
      float p0[8], p1[8], p2[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        uint32_t w0, w1, w2;
        split3_pair(x[c0 + 2 * q], x[c0 + 2 * q + 1], w0, w1, w2);
        p0[q] = __uint_as_float(w0);
        p1[q] = __uint_as_float(w1);
        p2[q] = __uint_as_float(w2);
      }
      const uint32_t col = TM_A + (uint32_t)(i0 + c0) / 2;
      tmem_st8(tmem + lane_base + col + 0 * 64, p0);
      tmem_st8(tmem + lane_base + col + 1 * 64, p1);
      tmem_st8(tmem + lane_base + col + 2 * 64, p2);
    }
    tmem_st_wait();
  };
  if (a.n > 0) write_pieces();

  const uint32_t idesc = idesc_f32acc(1, 1, 0, 0, 128, 128);
  const Tin *SK = static_cast<const Tin *>(a.seam_k);
  const Tin *SV = static_cast<const Tin *>(a.seam_v);
  const Tin *SQ = static_cast<const Tin *>(a.seam_q);
  uint32_t ph = 0;
  uint32_t dph = 0;  // phase of bar_d and bar_u (one completion each per seam token group)
  // bf16 seam tokens are exact B operands: their dot products with the state run on the tensor core
  constexpr bool TCD = std::is_same<Tin, __nv_bfloat16>::value;
  const bool kda = a.fam == HYPIC_FAM_KDA;
  const bool want_o = a.o_out != nullptr;
  // Tokens [t0, t0 + SG) of the seam window that follows composition step `st`, this thread's share,
  // as the stored values: nothing here uses a loaded register, so the loads stay in flight until
  // the values are stored to shared memory (after a block barrier, which no instruction crosses).
  auto load_seam = [&](int st, int t0, Tin (&lk)[NL], Tin (&lv)[NL], Tin (&lq)[NL], float (&lg)[NL], float &la,
                       float &lb) {
    const int ng = a.w - t0 < SG ? a.w - t0 : SG;
    const size_t tok0 = ((size_t)b * (a.n - 1) + st) * a.w + t0;
    la = 1.f;
    lb = 0.f;
    if (tid < ng) {
      const size_t tok = tok0 + tid;
      if (a.fam == HYPIC_FAM_GATED_DELTA) la = a.seam_alpha[tok * H + h];
      lb = a.seam_beta[tok * H + h];
    }
#pragma unroll
    for (int it = 0; it < NL; ++it) {
      const int e = tid + it * NT, t = e / D, i = e % D;
      lk[it] = lv[it] = lq[it] = Tin(0.f);
      lg[it] = 1.f;
      if (t < ng) {
        const size_t g = ((tok0 + t) * H + h) * D + i;
        lk[it] = SK[g];
        lv[it] = SV[g];
        if (want_o) lq[it] = SQ[g];
        if (kda) lg[it] = a.seam_alpha[g];
      }
    }
  };

  for (int step = 0; step < a.n; ++step) {
    // (1) T of this step: fp32 staging -> three bf16 B pieces [128 i][128 k], K-major, swizzled.
    // Thread (row i, half) converts k in [64 half, 64 half + 64).  bf16 pairs: already in place.
    if (tid == 0) {
      const bool got = PB ? mbar_wait_cycles(&bar_t[step & 1], (uint32_t)(step >> 1) & 1u, a.err)
                          : mbar_wait_cycles(&bar_t[0], ph, a.err);
      if (!got) abort_flag = 1;
    }
    tc_fence_before();
    __syncthreads();
    if (abort_flag) break;
    if (!PB) {
      const uint32_t i = (uint32_t)j;
#pragma unroll
      for (int kq = 0; kq < 2; ++kq) {
        const int kb = half * 2 + kq;  // 32-wide staging box
#pragma unroll
        for (int cp = 0; cp < 4; ++cp) {  // 8 consecutive k = 32 kb + 8 cp
          const float4 u = *reinterpret_cast<const float4 *>(sm + OFF_TST + kb * 16384 + sw128_offset(i, 2 * cp));
          const float4 w4 =
              *reinterpret_cast<const float4 *>(sm + OFF_TST + kb * 16384 + sw128_offset(i, 2 * cp + 1));
          uint32_t q0[4], q1[4], q2[4];
          split3_pair(u.x, u.y, q0[0], q1[0], q2[0]);
          split3_pair(u.z, u.w, q0[1], q1[1], q2[1]);
          split3_pair(w4.x, w4.y, q0[2], q1[2], q2[2]);
          split3_pair(w4.z, w4.w, q0[3], q1[3], q2[3]);
          const uint32_t chunk = ((uint32_t)(kb & 1) << 2) + (uint32_t)cp;
          const uint32_t off = (uint32_t)half * 16384 + sw128_offset(i, chunk);
          *reinterpret_cast<uint4 *>(sm + OFF_TB + 0 * 32768 + off) = make_uint4(q0[0], q0[1], q0[2], q0[3]);
          *reinterpret_cast<uint4 *>(sm + OFF_TB + 1 * 32768 + off) = make_uint4(q1[0], q1[1], q1[2], q1[3]);
          *reinterpret_cast<uint4 *>(sm + OFF_TB + 2 * 32768 + off) = make_uint4(q2[0], q2[1], q2[2], q2[3]);
        }
      }
    }
    if (!PB) {
      fence_proxy_async();  // B pieces are read by the MMA; the staging buffer is refilled by TMA
      tc_fence_before();
      __syncthreads();
    }
    // The first token group of the seam window after this step is loaded now: the state lives in
    // tensor memory until the epilogue, so these registers are free, and the loads' latency hides
    // behind the step's products.
    Tin pk[NL], pv[NL], pq[NL];
    float pg[NL], pa = 1.f, pb = 0.f;
    if (a.w > 0 && step + 1 < a.n) load_seam(step, 0, pk, pv, pq, pg, pa, pb);
    if (tid == 0) {
      tc_fence_after();
      // fp32: the staging buffer is consumed.  bf16: the other buffer's MMAs (step - 1) are done.
      if (step + 1 < a.n) issue_T(step + 1);
      if (PB) {
        // (2) D = S^T T^T with three products (A piece, exact T), smallest first: lo, mid, hi.
#pragma unroll
        for (int pr = 0; pr < 3; ++pr) {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t bo = OFF_TB16 + (step & 1) * 32768 + (kk >> 2) * 16384 + (kk & 3) * 32;
            mma_f16_tmem_a(tmem + TM_D, tmem + TM_A + (2 - pr) * 64 + kk * 8, sdesc_sw128(sb + bo, 16, 1024),
                           idesc, (pr | kk) != 0);
          }
        }
      } else {
        // (2) D = S^T T^T with six split products (A piece, B piece), smallest first:
        // (2,0) (1,1) (0,2) (1,0) (0,1) (0,0).
        const int pa[6] = {2, 1, 0, 1, 0, 0}, pb[6] = {0, 1, 2, 0, 1, 0};
#pragma unroll
        for (int pr = 0; pr < 6; ++pr) {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t bo = OFF_TB + pb[pr] * 32768 + (kk >> 2) * 16384 + (kk & 3) * 32;
            mma_f16_tmem_a(tmem + TM_D, tmem + TM_A + pa[pr] * 64 + kk * 8, sdesc_sw128(sb + bo, 16, 1024),
                           idesc, (pr | kk) != 0);
          }
        }
      }
      mma_commit(&bar_m);
    }
    // While the MMAs run, every thread loads its rows of S_{C|0} column j into x (the state itself
    // now lives in tensor memory as the A pieces, so x is free).
    if (addend) {
      int got = 1;
      if ((tid & 31) == 0) got = mbar_wait_cycles(&bar_s, ph, a.err) ? 1 : 0;
      __syncwarp();
      got = __shfl_sync(0xffffffffu, got, 0);
      if (!got) abort_flag = 1;
      if (PB) {
        const __nv_bfloat16 *s0b = reinterpret_cast<const __nv_bfloat16 *>(sS0);
#pragma unroll
        for (int r = 0; r < R; ++r) x[r] = __bfloat162float(s0b[(i0 + r) * D + j]);
      } else {
#pragma unroll
        for (int r = 0; r < R; ++r) x[r] = sS0[(i0 + r) * D + j];
      }
    } else {
#pragma unroll
      for (int r = 0; r < R; ++r) x[r] = 0.f;
    }
    if (tid == 0 && !mbar_wait_cycles(&bar_m, ph, a.err)) abort_flag = 1;
    __syncthreads();
    tc_fence_after();
    if (abort_flag) break;

    // (3) Epilogue: rows i0.. of column j of S_new = D row j + S_{C|0}.
#pragma unroll
    for (int hb = 0; hb < R; hb += 32) {
      float dv[32];
      tmem_ld32(tmem + lane_base + TM_D + i0 + hb, dv);
#pragma unroll
      for (int r = 0; r < 32; ++r) x[hb + r] += dv[r];
    }
    if (a.scan) {
      float *rec = (isT ? a.T_rec : a.S_rec) + ((size_t)step * H + h) * D * D;
#pragma unroll
      for (int r = 0; r < R; ++r) rec[(size_t)(i0 + r) * D + j] = x[r];
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();  // S0 staging is consumed
    if (step + 1 < a.n) {
      // (4) Seam tokens of the next segment, token by token on the register column: gate first
      // (a_t, 1, or KDA's per-channel g_t), y = gate * x, then x = y + b (v_j - k . y) k and
      // o_j = q . x = q . y + b (v_j - k . y) (q . k).  The S0 staging buffer is free here: a
      // group of up to SG tokens lands in it in one coalesced pass (one memory latency per group),
      // one warp per token forms q . k, and each token then needs a single barrier, the partial
      // sums k . y and q . y of the two row halves alternating between two slots.
      if (a.w > 0) {
        float *sK = sS0;               // [SG][D]
        float *sQ = sK + SG * D;       // [SG][D]
        float *sV = sQ + SG * D;       // [SG][D]
        float *sGc = sV + SG * D;      // [SG][D], KDA channel gates
        float *sA = sGc + SG * D;      // [SG] scalar gates
        float *sB = sA + SG;           // [SG]
        float *sQK = sB + SG;          // [SG]
        float *redk = sQK + SG;        // [2][2][D]
        float *redq = redk + 4 * D;    // [2][2][D]
        for (int t0 = 0; t0 < a.w; t0 += SG) {
          const int ng = a.w - t0 < SG ? a.w - t0 : SG;
          const size_t tok0 = ((size_t)b * (a.n - 1) + step) * a.w + t0;
          {
            // the first group was loaded at the top of the step; later groups load here, all of a
            // group's loads issued before the first store (one memory latency)
            Tin lk[NL], lv[NL], lq[NL];
            float lg[NL], la, lb;
            if (t0 == 0) {
#pragma unroll
              for (int it = 0; it < NL; ++it) {
                lk[it] = pk[it];
                lv[it] = pv[it];
                lq[it] = pq[it];
                lg[it] = pg[it];
              }
              la = pa;
              lb = pb;
            } else {
              load_seam(step, t0, lk, lv, lq, lg, la, lb);
            }
#pragma unroll
            for (int it = 0; it < NL; ++it) {
              const int e = tid + it * NT;
              if (e / D < ng) {
                sK[e] = to_f32<Tin>(lk[it]);
                sV[e] = to_f32<Tin>(lv[it]);
                sQ[e] = to_f32<Tin>(lq[it]);
                sGc[e] = lg[it];
              }
            }
            if (tid < ng) {
              sA[tid] = la;
              sB[tid] = lb;
            }
          }
          __syncthreads();
          if (!kda) {
            // Scalar gates: the group in chunked form.  With D_ts = a_{s+1} ... a_t (s < t; D_tt = 1;
            // gamma_t = a_0 ... a_t), u_t = k_t . x and p_t = q_t . x for the column x on entry, the
            // effective writes w solve (I + L) w = b (v - gamma u), L_ts = b_t D_ts (k_t . k_s)
            // (s < t); then o_t = gamma_t p_t + sum_{s <= t} D_ts (q_t . k_s) w_s and
            // x <- gamma_last x + sum_s D_last,s w_s k_s.  Decay factors are products of gates,
            // never quotients.
            float *sL = redq + 4 * D;   // [SG][SG]: L (s < t), D (s >= t unused)
            float *sM = sL + SG * SG;   // [SG][SG]: D_ts (q_t . k_s), s <= t
            float *sGam = sM + SG * SG; // [SG]: gamma_t
            float *sF = sGam + SG;      // [SG]: D_last,s
            float *sU = sF + SG;        // [2 halves][SG][D]: partial k_t . x, then q_t . x
            if constexpr (TCD) {
              // u_t = k_t . S_j and p_t = q_t . S_j for every column j at once: D = S^T [K; Q]^T
              // (M = 128 columns j, N = 16, K = 128 rows i) against the state's exact three A pieces,
              // written to tensor memory now; B holds k_t in rows 0..7 and q_t in rows 8..15 (exact
              // bf16, zero past the group), K-major and swizzled.  The warps form the Gram meanwhile.
              uint8_t *bt = reinterpret_cast<uint8_t *>(sS0) + SEAM_BT;
              {
                const int r = tid >> 4, c = tid & 15, t = r & 7;
                const bool isq = r >= SG;
                float v8[8];
                const bool live = t < ng && (!isq || want_o);
                const float *src = (isq ? sQ : sK) + t * D + 8 * c;
#pragma unroll
                for (int e = 0; e < 8; ++e) v8[e] = live ? src[e] : 0.f;
                uint32_t w4[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const __nv_bfloat162 p2 = __floats2bfloat162_rn(v8[2 * e], v8[2 * e + 1]);
                  w4[e] = *reinterpret_cast<const uint32_t *>(&p2);
                }
                *reinterpret_cast<uint4 *>(bt + (c >> 3) * 2048 + sw128_offset((uint32_t)r, (uint32_t)(c & 7))) =
                    make_uint4(w4[0], w4[1], w4[2], w4[3]);
              }
              write_pieces();
              fence_proxy_async();
              tc_fence_before();
              __syncthreads();
              if (tid == 0) {
                tc_fence_after();
                const uint32_t id16 = idesc_f32acc(1, 1, 0, 0, 128, 16);
                const uint32_t bb = smem_u32(bt);
#pragma unroll
                for (int pr = 0; pr < 3; ++pr) {
#pragma unroll
                  for (int kk = 0; kk < 8; ++kk)
                    mma_f16_tmem_a(tmem + TM_DOT, tmem + TM_A + (2 - pr) * 64 + kk * 8,
                                   sdesc_sw128(bb + (kk >> 2) * 2048 + (kk & 3) * 32, 16, 1024), id16,
                                   (pr | kk) != 0);
                }
                mma_commit(&bar_d);
              }
            }
            if (warp < ng) {
              // warp t: (k_t . k_s) and (q_t . k_s) for s < ng, and row t of the decay products
              const int t = warp, ln = tid & 31;
              float gk[SG], gq[SG];
#pragma unroll
              for (int s2 = 0; s2 < SG; ++s2) {
                gk[s2] = 0.f;
                gq[s2] = 0.f;
              }
#pragma unroll
              for (int i = ln; i < D; i += 32) {
                const float kt = sK[t * D + i], qt = want_o ? sQ[t * D + i] : 0.f;
#pragma unroll
                for (int s2 = 0; s2 < SG; ++s2) {
                  if (s2 < ng) {
                    const float ks = sK[s2 * D + i];
                    gk[s2] = fmaf(kt, ks, gk[s2]);
                    gq[s2] = fmaf(qt, ks, gq[s2]);
                  }
                }
              }
#pragma unroll
              for (int s2 = 0; s2 < SG; ++s2) {
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                  gk[s2] += __shfl_xor_sync(0xffffffffu, gk[s2], o);
                  gq[s2] += __shfl_xor_sync(0xffffffffu, gq[s2], o);
                }
              }
              if (ln == 0) {
                float dts = 1.f;  // D_ts for s = t, t - 1, ...
#pragma unroll
                for (int s2 = SG - 1; s2 >= 0; --s2) {
                  if (s2 <= t) {
                    sM[t * SG + s2] = dts * gq[s2];
                    if (s2 < t) sL[t * SG + s2] = sB[t] * dts * gk[s2];
                    dts *= sA[s2];
                  }
                }
                sGam[t] = dts;  // a_0 ... a_t
                if (t == ng - 1) {
                  float f = 1.f;
                  for (int s2 = t; s2 >= 0; --s2) {
                    sF[s2] = f;
                    f *= sA[s2];
                  }
                }
              }
            }
            float wv[SG];
            if constexpr (TCD) {
              float dd[16];
              int got = 1;
              if ((tid & 31) == 0) got = mbar_wait_cycles(&bar_d, dph, a.err) ? 1 : 0;
              __syncwarp();
              if (!__shfl_sync(0xffffffffu, got, 0)) abort_flag = 1;
              tc_fence_after();
              tmem_ld16(tmem + lane_base + TM_DOT, dd);
              __syncthreads();  // the Gram's rows are complete
#pragma unroll
              for (int t = 0; t < SG; ++t) {
                if (t < ng) {
                  float acc = sB[t] * (sV[t * D + j] - sGam[t] * dd[t]);
#pragma unroll
                  for (int s2 = 0; s2 < t; ++s2) acc = fmaf(-sL[t * SG + s2], wv[s2], acc);
                  wv[t] = acc;
                }
              }
              if (want_o && half == 0) {
#pragma unroll
                for (int t = 0; t < SG; ++t) {
                  if (t < ng) {
                    float o = sGam[t] * dd[SG + t];
#pragma unroll
                    for (int s2 = 0; s2 <= t; ++s2) o = fmaf(sM[t * SG + s2], wv[s2], o);
                    a.o_out[((tok0 + t) * H + h) * D + j] = o;
                  }
                }
              }
            } else {
            // partial dot products of this thread's 64 rows
            {
              float u[SG];
#pragma unroll
              for (int t = 0; t < SG; ++t) u[t] = 0.f;
#pragma unroll
              for (int r = 0; r < R; r += 4) {
#pragma unroll
                for (int t = 0; t < SG; ++t) {
                  if (t < ng) {
                    const float4 k4 = *reinterpret_cast<const float4 *>(sK + t * D + i0 + r);
                    u[t] = fmaf(k4.x, x[r], u[t]);
                    u[t] = fmaf(k4.y, x[r + 1], u[t]);
                    u[t] = fmaf(k4.z, x[r + 2], u[t]);
                    u[t] = fmaf(k4.w, x[r + 3], u[t]);
                  }
                }
              }
#pragma unroll
              for (int t = 0; t < SG; ++t)
                if (t < ng) sU[(half * SG + t) * D + j] = u[t];
            }
            __syncthreads();
            {
              float uk[SG];
#pragma unroll
              for (int t = 0; t < SG; ++t)
                if (t < ng) uk[t] = sU[t * D + j] + sU[(SG + t) * D + j];
#pragma unroll
              for (int t = 0; t < SG; ++t) {
                if (t < ng) {
                  float acc = sB[t] * (sV[t * D + j] - sGam[t] * uk[t]);
#pragma unroll
                  for (int s2 = 0; s2 < t; ++s2) acc = fmaf(-sL[t * SG + s2], wv[s2], acc);
                  wv[t] = acc;
                }
              }
            }
            if (want_o) {
              __syncthreads();  // sU is reused for q . x
              float pq[SG];
#pragma unroll
              for (int t = 0; t < SG; ++t) pq[t] = 0.f;
#pragma unroll
              for (int r = 0; r < R; r += 4) {
#pragma unroll
                for (int t = 0; t < SG; ++t) {
                  if (t < ng) {
                    const float4 q4 = *reinterpret_cast<const float4 *>(sQ + t * D + i0 + r);
                    pq[t] = fmaf(q4.x, x[r], pq[t]);
                    pq[t] = fmaf(q4.y, x[r + 1], pq[t]);
                    pq[t] = fmaf(q4.z, x[r + 2], pq[t]);
                    pq[t] = fmaf(q4.w, x[r + 3], pq[t]);
                  }
                }
              }
#pragma unroll
              for (int t = 0; t < SG; ++t)
                if (t < ng) sU[(half * SG + t) * D + j] = pq[t];
              __syncthreads();
              if (half == 0) {
#pragma unroll
                for (int t = 0; t < SG; ++t) {
                  if (t < ng) {
                    float o = sGam[t] * (sU[t * D + j] + sU[(SG + t) * D + j]);
#pragma unroll
                    for (int s2 = 0; s2 <= t; ++s2) o = fmaf(sM[t * SG + s2], wv[s2], o);
                    a.o_out[((tok0 + t) * H + h) * D + j] = o;
                  }
                }
              }
            }
            }
            // x <- gamma_last x + sum_s D_last,s w_s k_s
            if constexpr (TCD) {
              // On the tensor core: D = C^T K over the group's tokens (K = 16, the rows past the
              // group contribute zero), A = C^T with C_s[j] = D_last,s w_s[j] in its exact three-way
              // split (tensor memory, written by one thread per column), B = the key rows of the dot
              // products' B tile read as an MN-major operand (rows s, columns i).
              const float gl = sGam[ng - 1];
              if (half == 0) {
                float c0[8], c1[8], c2[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                  const int s0 = 2 * q, s1 = 2 * q + 1;
                  const float ca = (s0 < SG && s0 < ng) ? sF[s0] * wv[s0 < SG ? s0 : 0] : 0.f;
                  const float cb = (s1 < SG && s1 < ng) ? sF[s1] * wv[s1 < SG ? s1 : 0] : 0.f;
                  uint32_t w0, w1, w2;
                  split3_pair(ca, cb, w0, w1, w2);
                  c0[q] = __uint_as_float(w0);
                  c1[q] = __uint_as_float(w1);
                  c2[q] = __uint_as_float(w2);
                }
                tmem_st8(tmem + lane_base + TM_C, c0);
                tmem_st8(tmem + lane_base + TM_C + 8, c1);
                tmem_st8(tmem + lane_base + TM_C + 16, c2);
                tmem_st_wait();
              }
              tc_fence_before();
              __syncthreads();
              if (tid == 0) {
                tc_fence_after();
                const uint32_t idU = idesc_f32acc(1, 1, 0, 1, 128, 128);
                const uint64_t bK = sdesc_sw128(smem_u32(reinterpret_cast<uint8_t *>(sS0) + SEAM_BT), 2048, 1024);
#pragma unroll
                for (int pr = 0; pr < 3; ++pr) mma_f16_tmem_a(tmem + TM_D, tmem + TM_C + (2 - pr) * 8, bK, idU, pr > 0);
                mma_commit(&bar_u);
              }
              int got = 1;
              if ((tid & 31) == 0) got = mbar_wait_cycles(&bar_u, dph, a.err) ? 1 : 0;
              __syncwarp();
              if (!__shfl_sync(0xffffffffu, got, 0)) abort_flag = 1;
              tc_fence_after();
#pragma unroll
              for (int hb = 0; hb < R; hb += 32) {
                float dv[32];
                tmem_ld32(tmem + lane_base + TM_D + i0 + hb, dv);
#pragma unroll
                for (int r = 0; r < 32; ++r) x[hb + r] = fmaf(gl, x[hb + r], dv[r]);
              }
            } else {
              const float gl = sGam[ng - 1];
              float cs[SG];
#pragma unroll
              for (int t = 0; t < SG; ++t) cs[t] = t < ng ? sF[t] * wv[t] : 0.f;
#pragma unroll
              for (int r = 0; r < R; r += 4) {
                float v0 = gl * x[r], v1 = gl * x[r + 1], v2 = gl * x[r + 2], v3 = gl * x[r + 3];
#pragma unroll
                for (int t = 0; t < SG; ++t) {
                  if (t < ng) {
                    const float4 k4 = *reinterpret_cast<const float4 *>(sK + t * D + i0 + r);
                    v0 = fmaf(cs[t], k4.x, v0);
                    v1 = fmaf(cs[t], k4.y, v1);
                    v2 = fmaf(cs[t], k4.z, v2);
                    v3 = fmaf(cs[t], k4.w, v3);
                  }
                }
                x[r] = v0;
                x[r + 1] = v1;
                x[r + 2] = v2;
                x[r + 3] = v3;
              }
            }
          } else {
            if (want_o && warp < ng) {
              float acc = 0.f;
#pragma unroll
              for (int i = (tid & 31); i < D; i += 32) acc = fmaf(sQ[warp * D + i], sK[warp * D + i], acc);
#pragma unroll
              for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
              if ((tid & 31) == 0) sQK[warp] = acc;
            }
            for (int t = 0; t < ng; ++t) {
              const int sl = t & 1;
              const float *sk = sK + t * D, *sq = sQ + t * D;
              if (kda) {
#pragma unroll
                for (int r = 0; r < R; ++r) x[r] *= sGc[t * D + i0 + r];
              } else {
                const float at = sA[t];
#pragma unroll
                for (int r = 0; r < R; ++r) x[r] *= at;
              }
              float c0 = 0.f, c1 = 0.f;
#pragma unroll
              for (int r = 0; r < R; r += 2) {
                c0 = fmaf(sk[i0 + r], x[r], c0);
                c1 = fmaf(sk[i0 + r + 1], x[r + 1], c1);
              }
              redk[(sl * 2 + half) * D + j] = c0 + c1;
              if (want_o) {
                float e0 = 0.f, e1 = 0.f;
#pragma unroll
                for (int r = 0; r < R; r += 2) {
                  e0 = fmaf(sq[i0 + r], x[r], e0);
                  e1 = fmaf(sq[i0 + r + 1], x[r + 1], e1);
                }
                redq[(sl * 2 + half) * D + j] = e0 + e1;
              }
              __syncthreads();
              const float kx = redk[sl * 2 * D + j] + redk[(sl * 2 + 1) * D + j];
              const float coef = sB[t] * (sV[t * D + j] - kx);
#pragma unroll
              for (int r = 0; r < R; ++r) x[r] = fmaf(coef, sk[i0 + r], x[r]);
              if (want_o && half == 0) {
                const float qy = redq[sl * 2 * D + j] + redq[(sl * 2 + 1) * D + j];
                a.o_out[((tok0 + t) * H + h) * D + j] = qy + coef * sQK[t];
              }
            }
          }
          __syncthreads();  // the group's tokens are consumed
          if (TCD && !kda) dph ^= 1u;
        }
        fence_proxy_async();  // the buffer is refilled by TMA next
        __syncthreads();
      }
      if (tid == 0 && addend) issue_S(step + 1);
      write_pieces();
    }
    ph ^= 1u;
  }

  if (!abort_flag && !a.scan) {
    float *out = a.S_out + base_bh;
#pragma unroll
    for (int r = 0; r < R; ++r) out[(size_t)(i0 + r) * D + j] = x[r];
  }
  if (abort_flag && tid == 0) {
    mbar_wait_cycles(&bar_m, ph, nullptr, 200000000LL);
    if (TCD) {
      mbar_wait_cycles(&bar_d, dph, nullptr, 200000000LL);
      mbar_wait_cycles(&bar_u, dph, nullptr, 200000000LL);
    }
    mbar_wait_cycles(&bar_t[0], PB ? 0u : ph, nullptr, 200000000LL);
    if (PB) {
      mbar_wait_cycles(&bar_t[0], 1u, nullptr, 200000000LL);
      mbar_wait_cycles(&bar_t[1], 0u, nullptr, 200000000LL);
      mbar_wait_cycles(&bar_t[1], 1u, nullptr, 200000000LL);
    }
    mbar_wait_cycles(&bar_s, ph, nullptr, 200000000LL);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, TM_COLS);
}

}  // namespace

bool compose_tc_supported(int D_, int fam) {
  return D_ == D && (fam == HYPIC_FAM_DELTA || fam == HYPIC_FAM_GATED_DELTA || fam == HYPIC_FAM_KDA);
}

template <typename Tin, bool PB>
cudaError_t launch_one(const CUtensorMap &mT, const CUtensorMap &mS, const ComposeTcArgs &a, long long blocks,
                       cudaStream_t st) {
  const uint32_t smem = PB ? SMEM_BYTES16 : SMEM_BYTES;
  cudaError_t e = cudaFuncSetAttribute(compose_tc_kernel<Tin, PB>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  compose_tc_kernel<Tin, PB><<<(unsigned)blocks, NT, smem, st>>>(mT, mS, a);
  return cudaGetLastError();
}

cudaError_t launch_compose_pipe(const CUtensorMap &mT, const CUtensorMap &mS, int H, int B, int n,
                                const int32_t *idx, int64_t pool_size, const float *S_init, float *S_out, int *err,
                                cudaStream_t st);

cudaError_t launch_compose_pipe32(int H, int B, int n, const int32_t *idx, int64_t pool_size, const float *pool_T,
                                  const float *pool_S, const float *S_init, float *S_out, int *err, cudaStream_t st);
cudaError_t launch_scan_pipe32(int H, int n, const float *T, const float *S, float *Tp, float *Sp, void *ws,
                               size_t ws_bytes, int *err, cudaStream_t st);

cudaError_t launch_compose_tc(const ChainArgs &c, cudaStream_t st) {
  const uint64_t rows = (uint64_t)c.pool_size * c.H * D;
  if (rows >= ((uint64_t)1 << 31)) return cudaErrorInvalidValue;
  const bool pb = c.pair_bf16 != 0;
  if (!pb && c.w == 0 && c.scan)
    return launch_scan_pipe32(c.H, c.n, static_cast<const float *>(c.pool_T), static_cast<const float *>(c.pool_S),
                              c.T_rec, c.S_rec, c.ws, c.ws_bytes, c.err, st);
  if (!pb && c.w == 0)
    return launch_compose_pipe32(c.H, c.B, c.n, c.idx, c.pool_size, static_cast<const float *>(c.pool_T),
                                 static_cast<const float *>(c.pool_S), c.S_init, c.S_out, c.err, st);
  CUtensorMap mT, mS;
  if (pb) {
    if (!make_tmap_bf16_2d(&mT, c.pool_T, rows, D, D, 64, 128)) return cudaErrorInvalidValue;
  } else if (!make_tmap_f32_2d(&mT, c.pool_T, rows, D, D, 32, 128)) {
    return cudaErrorInvalidValue;
  }
  {
    // S_{C|0} as one [128][128] box, no swizzle, row-major in shared memory.
    auto fn = tma_encode_fn();
    if (!fn) return cudaErrorInvalidValue;
    const uint32_t es = pb ? 2 : 4;
    cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)D * es};
    cuuint32_t box[2] = {128, 128};
    cuuint32_t estr[2] = {1, 1};
    if (fn(&mS, pb ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
           const_cast<void *>(c.pool_S), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
           CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  if (pb && !c.scan && c.w == 0)
    return launch_compose_pipe(mT, mS, c.H, c.B, c.n, c.idx, c.pool_size, c.S_init, c.S_out, c.err, st);
  ComposeTcArgs a{};
  a.H = c.H;
  a.B = c.B;
  a.n = c.n;
  a.w = c.w;
  a.B_major = 0;
  a.idx = c.idx;
  a.pool_size = c.pool_size;
  a.S_init = c.S_init;
  a.S_out = c.S_out;
  a.scan = c.scan;
  a.T_rec = c.T_rec;
  a.S_rec = c.S_rec;
  a.fam = c.fam;
  a.seam_bf16 = c.seam.in_dtype == HYPIC_BF16;
  a.seam_k = c.seam.k;
  a.seam_v = c.seam.v;
  a.seam_q = c.seam.q;
  a.seam_alpha = c.seam.alpha;
  a.seam_beta = c.seam.beta;
  a.o_out = c.o_out;
  a.err = c.err;
  const long long blocks = c.scan ? (long long)c.H * 2 : (long long)c.B * c.H;
  if (blocks <= 0) return cudaSuccess;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  if (a.seam_bf16) {
    return pb ? launch_one<__nv_bfloat16, true>(mT, mS, a, blocks, st)
              : launch_one<__nv_bfloat16, false>(mT, mS, a, blocks, st);
  }
  return pb ? launch_one<float, true>(mT, mS, a, blocks, st) : launch_one<float, false>(mT, mS, a, blocks, st);
}

}  // namespace hypic
