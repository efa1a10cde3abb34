// Pipelined tensor-core composition over pairs stored in bf16 (delta families, d = 128, no seam
// windows): S <- T_C S + S_{C|0} applied in prompt order (HYPIC reading notes, Method 2, paper
// Eq. (6)), with the cached pairs in 16-bit storage (Method 3, Table 3 sizes).
//
// The product is the transposed one the unpipelined chain uses, D = S_new^T = S^T T^T (M = 128
// columns j in the TMEM lanes, N = 128 rows i, K = 128), A = S^T as three exact bf16 pieces in
// tensor memory, B = T (exact bf16) straight from its TMA tile, three products (A piece x T),
// accumulated smallest first.  Thread (j, h) owns rows 64h .. 64h + 63 of column j: its epilogue
// reads output rows 64h.. (N half h) and writes the A pieces of contraction half h of the next
// step.  A step issues its products in this order:
//     lo and mid pieces, contraction half 0     (waits for half 0's pieces of the last step)
//     lo and mid pieces, contraction half 1     (waits for half 1's pieces)
//     hi piece, output half 0 (N = 64)  -> commit e0
//     hi piece, output half 1 (N = 64)  -> commit e1
// so half 0's epilogue runs beside the last products, and the next step's first products beside
// half 1's epilogue.  For that the accumulator and the hi piece are double buffered by step
// parity (the lo and mid pieces are no longer read once e0 has fired): 2 x 128 + 64 + 64 + 2 x 64
// = 512 columns.  The epilogue loads its S_{C|0} rows while it waits, and T and S_{C|0} arrive by
// TMA two steps ahead (three buffers).  A dedicated warp issues the MMAs and the copies; the
// epilogue threads signal it through mbarriers.
#include <cuda_bf16.h>

#include "tc_ptx.cuh"
#include "tma_host.h"

namespace hypic {
namespace {

using namespace tc;

constexpr int D = 128;
constexpr int NE = 256;       // epilogue threads: column j = tid & 127, row half h = tid >> 7
constexpr int NTH = NE + 32;  // + the control warp (MMA issue and TMA)
constexpr int R = 64;         // rows of a column each epilogue thread owns
constexpr int NBUF = 3;       // T and S_{C|0} buffers
constexpr uint32_t BUF_T = 32768;   // T: two k-blocks of [128 i][64 k] bf16, K-major, 128-byte swizzle
constexpr uint32_t BUF_S = 32768;   // S_{C|0}: [128 i][128 j] bf16, row-major
constexpr uint32_t OFF_T = 0, OFF_S = NBUF * BUF_T;
constexpr uint32_t SMEM_BYTES = OFF_S + NBUF * BUF_S + 1024;
// Tensor memory: the accumulator D and the hi piece of S^T (two buffers each, by step parity),
// the mid and lo pieces.
constexpr uint32_t TM_D = 0, TM_MID = 256, TM_LO = 320, TM_HI = 384, TM_COLS = 512;

struct PipeArgs {
  int H, B, n;
  const int32_t *idx;
  int64_t pool_size;
  const float *S_init;
  float *S_out;
  int *err;
};

// Exact three-way split of two fp32 values into bf16 pieces, two per 32-bit word (hi keeps the
// sign, the exponent and the top 7 stored bits; the remainder is exact in fp32 and is split the
// same way; the last remainder has at most 8 significant bits, so x = hi + mid + lo exactly).
__device__ __forceinline__ void split3(float a, float b, uint32_t &p0, uint32_t &p1, uint32_t &p2) {
  const uint32_t ua = __float_as_uint(a), ub = __float_as_uint(b);
  const float ra = a - __uint_as_float(ua & 0xFFFF0000u), rb = b - __uint_as_float(ub & 0xFFFF0000u);
  const uint32_t ura = __float_as_uint(ra), urb = __float_as_uint(rb);
  const float la = ra - __uint_as_float(ura & 0xFFFF0000u), lb = rb - __uint_as_float(urb & 0xFFFF0000u);
  p0 = __byte_perm(ua, ub, 0x7632);
  p1 = __byte_perm(ura, urb, 0x7632);
  p2 = __byte_perm(__float_as_uint(la), __float_as_uint(lb), 0x7632);
}

__device__ __forceinline__ void st8(uint32_t taddr, const uint32_t (&v)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
               "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
               : "memory");
}

__global__ void __launch_bounds__(NTH, 1)
    compose_pipe_kernel(const __grid_constant__ CUtensorMap mapT, const __grid_constant__ CUtensorMap mapS,
                        PipeArgs a) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar_t[NBUF], bar_s[NBUF];
  __shared__ uint64_t bar_e[2];        // MMA commits: output half 0 done, all done
  __shared__ uint64_t bar_a[2];        // epilogue of half h done (its A pieces written)
  __shared__ uint32_t tmem_slot;
  __shared__ volatile int abort_flag;
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(sm);
  const int tid = threadIdx.x, warp = tid >> 5;
  const int H = a.H, n = a.n;
  const int b = blockIdx.x % a.B, h = blockIdx.x / a.B;  // head-major: one head's requests together

  if (tid == 0) {
    for (int i = 0; i < NBUF; ++i) {
      mbar_init(&bar_t[i], 1);
      mbar_init(&bar_s[i], 1);
    }
    mbar_init(&bar_e[0], 1);
    mbar_init(&bar_e[1], 1);
    mbar_init(&bar_a[0], NE / 2);
    mbar_init(&bar_a[1], NE / 2);
    mbar_fence_init();
    abort_flag = 0;
  }
  if (warp == 0) {
    tmem_alloc(&tmem_slot, TM_COLS);
    tmem_relinquish();
  }
  const size_t base_bh = ((size_t)b * H + h) * D * D;
  const int j = tid & (D - 1), half = (tid >> 7) & 1, i0 = half * R;
  const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
  float x[R];
  if (tid < NE) {
#pragma unroll
    for (int r = 0; r < R; ++r) x[r] = a.S_init ? a.S_init[base_bh + (size_t)(i0 + r) * D + j] : 0.f;
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;

  // This thread's rows i0 .. i0 + 63 of column j as A pieces (contraction half `half`) of the step
  // with parity p.
  auto write_pieces = [&](uint32_t p) {
#pragma unroll
    for (int c0 = 0; c0 < R; c0 += 16) {
      uint32_t p0[8], p1[8], p2[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) split3(x[c0 + 2 * q], x[c0 + 2 * q + 1], p0[q], p1[q], p2[q]);
      const uint32_t col = tmem + lane_base + (uint32_t)(i0 + c0) / 2;
      st8(col + TM_HI + p * 64, p0);
      st8(col + TM_MID, p1);
      st8(col + TM_LO, p2);
    }
    tmem_st_wait();
  };
  if (tid < NE && n > 0) write_pieces(0);
  tc_fence_before();
  __syncthreads();

  if (warp == NE / 32) {
    // ---- control warp: lane 0 issues every copy and MMA -------------------------------------
    if ((tid & 31) == 0) {
      tc_fence_after();
      prefetch_tmap(&mapT);
      prefetch_tmap(&mapS);
      int loads = 0, commits = 0;
      auto entry = [&](int s) -> int64_t {
        int64_t p = a.idx ? (int64_t)a.idx[(size_t)b * n + s] : (int64_t)s;
        if (p < 0 || p >= a.pool_size) {
          set_error(a.err, HYPIC_EDEVICE);
          p = 0;
        }
        return p;
      };
      auto load = [&](int s) {
        const int bs = s % NBUF;
        const int row = (int)((entry(s) * H + h) * D);
        mbar_arrive_expect_tx(&bar_t[bs], BUF_T);
        tma_load_2d(sm + OFF_T + bs * BUF_T, &mapT, &bar_t[bs], 0, row);
        tma_load_2d(sm + OFF_T + bs * BUF_T + 16384, &mapT, &bar_t[bs], 64, row);
        mbar_arrive_expect_tx(&bar_s[bs], BUF_S);
        tma_load_2d(sm + OFF_S + bs * BUF_S, &mapS, &bar_s[bs], 0, row);
        ++loads;
      };
      const uint32_t id128 = idesc_f32acc(1, 1, 0, 0, 128, 128), id64 = idesc_f32acc(1, 1, 0, 0, 128, 64);
      // Products of the A piece at column `pc` with T over contraction half kh (four k-blocks of
      // 16) into D.
      auto prod = [&](uint32_t dt, int bs, uint32_t pc, int kh, bool first) {
        const uint32_t tb = sb + OFF_T + bs * BUF_T + kh * 16384;
        const uint32_t ak = tmem + pc + kh * 32;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_f16_tmem_a(dt, ak + kk * 8, sdesc_sw128(tb + kk * 32, 16, 1024), id128, (first && kk == 0) ? 0u : 1u);
      };
      // The hi piece's products for output half nh (rows 64 nh .. of T), both contraction halves.
      auto prod_hi = [&](uint32_t dt, int bs, uint32_t hc, int nh) {
#pragma unroll
        for (int kh = 0; kh < 2; ++kh) {
          const uint32_t tb = sb + OFF_T + bs * BUF_T + kh * 16384 + nh * 8192;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_f16_tmem_a(dt + nh * 64, tmem + hc + kh * 32 + kk * 8, sdesc_sw128(tb + kk * 32, 16, 1024), id64, 1u);
        }
      };
      bool pending = false;  // products issued since the last commit
      for (int s = 0; s < n && s < NBUF - 1; ++s) load(s);
      for (int s = 0; s < n; ++s) {
        const int bs = s % NBUF;
        const uint32_t pp = (uint32_t)(s - 1) & 1u;
        const uint32_t dt = tmem + TM_D + (uint32_t)(s & 1) * 128;
        bool ok = mbar_wait_cycles(&bar_t[bs], (uint32_t)(s / NBUF) & 1u, a.err);
        if (ok && s > 0) ok = mbar_wait_cycles(&bar_a[0], pp, a.err);
        if (!ok || abort_flag) {
          abort_flag = 1;
          break;
        }
        tc_fence_after();
        const uint32_t hc = TM_HI + (uint32_t)(s & 1) * 64;
        prod(dt, bs, TM_LO, 0, true);
        prod(dt, bs, TM_MID, 0, false);
        pending = true;
        if (s > 0 && !mbar_wait_cycles(&bar_a[1], pp, a.err)) {
          abort_flag = 1;
          break;
        }
        tc_fence_after();
        // step s - 1 is consumed whole: its buffers take step s + NBUF - 1
        if (s + NBUF - 1 < n) load(s + NBUF - 1);
        prod(dt, bs, TM_LO, 1, false);
        prod(dt, bs, TM_MID, 1, false);
        prod_hi(dt, bs, hc, 0);
        mma_commit(&bar_e[0]);
        prod_hi(dt, bs, hc, 1);
        mma_commit(&bar_e[1]);
        pending = false;
        ++commits;
      }
      if (pending) {
        mma_commit(&bar_e[1]);
        ++commits;
      }
      // Drain (bounded): every copy issued has landed and every product has completed before the
      // block's shared and tensor memory go away.
      if (commits > 0) mbar_wait_cycles(&bar_e[1], (uint32_t)(commits - 1) & 1u, nullptr, 200000000LL);
      for (int s = loads - NBUF > 0 ? loads - NBUF : 0; s < loads; ++s) {
        mbar_wait_cycles(&bar_t[s % NBUF], (uint32_t)(s / NBUF) & 1u, nullptr, 200000000LL);
        mbar_wait_cycles(&bar_s[s % NBUF], (uint32_t)(s / NBUF) & 1u, nullptr, 200000000LL);
      }
    }
  } else {
    // ---- epilogue threads: output half `half`, rows i0 .. i0 + 63 of column j ------------------
    const __nv_bfloat16 *s0 = reinterpret_cast<const __nv_bfloat16 *>(sm + OFF_S) + (size_t)i0 * D + j;
    // x = this thread's rows of S_{C|0} of step s (loaded while the products run)
    auto load_s0 = [&](int s) -> bool {
      int ok = 1;
      if ((tid & 31) == 0) {
        ok = !abort_flag && mbar_wait_cycles(&bar_s[s % NBUF], (uint32_t)(s / NBUF) & 1u, a.err);
        if (!ok) abort_flag = 1;
      }
      if (!__shfl_sync(0xffffffffu, ok, 0)) return false;
      const __nv_bfloat16 *sc = s0 + (size_t)(s % NBUF) * (BUF_S / 2);
#pragma unroll
      for (int r = 0; r < R; ++r) x[r] = __bfloat162float(sc[(size_t)r * D]);
      return true;
    };
    bool live = n > 0 ? load_s0(0) : true;
    // bounded wait of the warp on one of the commit barriers
    auto wait_e = [&](int k, int s) -> bool {
      int ok = 1;
      if ((tid & 31) == 0) {
        ok = !abort_flag && mbar_wait_cycles(&bar_e[k], (uint32_t)s & 1u, a.err);
        if (!ok) abort_flag = 1;
      }
      return __shfl_sync(0xffffffffu, ok, 0) != 0;
    };
    for (int s = 0; s < n && live; ++s) {
      if (!wait_e(half, s)) {
        live = false;
        break;
      }
      tc_fence_after();
      const uint32_t dt = tmem + lane_base + TM_D + (uint32_t)(s & 1) * 128 + i0;
#pragma unroll
      for (int hb = 0; hb < R; hb += 32) {
        float dv[32];
        tmem_ld32(dt + hb, dv);
#pragma unroll
        for (int r = 0; r < 32; ++r) x[hb + r] += dv[r];
      }
      if (s + 1 < n) {
        write_pieces((uint32_t)(s + 1) & 1u);
        fence_proxy_async();  // the S_{C|0} buffer is refilled by TMA after this arrival
        tc_fence_before();
        mbar_arrive(&bar_a[half]);
        live = load_s0(s + 1);
      }
    }
    if (live && !abort_flag) {
      float *out = a.S_out + base_bh;
#pragma unroll
      for (int r = 0; r < R; ++r) out[(size_t)(i0 + r) * D + j] = x[r];
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, TM_COLS);
  }
}

// ---- fp32 pairs: compose and the affine scan -------------------------------------------------
// With fp32 pairs T is not an exact bf16 operand: each step splits it into three exact bf16
// B pieces (hi, mid, lo), and the product takes the six terms (A piece a, B piece b) with
// a + b <= 2, smallest first.  The 256 epilogue threads also split T: warp w takes rows
// w, w + 8, .., lane l columns 4l .. 4l + 3 (one coalesced 512-byte row per warp and load), and
// they split the next step's T while this step's products run, into the other of two B buffers
// (2 x 96 KB of shared memory).  S_{C|0} comes straight from global memory into the registers
// of the thread that adds it, loaded while the products run.  A step issues
//     the five smaller terms over contraction half 0   (waits for half 0's A pieces)
//     the five smaller terms over contraction half 1   (waits for half 1's A pieces)
//     hi.hi, output half 0 (N = 64)  -> commit e0
//     hi.hi, output half 1 (N = 64)  -> commit e1, and the step's B buffer is free
// as the bf16-pair kernel does.  In scan mode (one block per head and column half of the
// augmented state [T | S], as the unpipelined chain has it) every step's state is written out.
// The scan may be cut into P chunks of m pairs (one block pair per chunk and head): a chunk then
// starts from a given carry state instead of [I | 0], and either writes every prefix at its global
// row or only its last one (the chunk's total) to a separate array; the two-level scan below
// combines these.
constexpr uint32_t BUF_B = 3 * 32768;          // B pieces of one T: hi, mid, lo x two k-blocks
constexpr uint32_t SMEM32 = 2 * BUF_B + 1024;  // two buffers by step parity

struct Pipe32Args {
  int H, B, n;
  const int32_t *idx;
  int64_t pool_size;
  const float *pool_T, *pool_S;
  const float *S_init;
  float *S_out;
  int scan;
  float *T_rec, *S_rec;
  int *err;
};
// Scan chunks: chunk c covers pairs [c m, min(n, c m + m)); chunk c > 0 starts from the carry
// (Tc, Sc)[c - 1] when Tc is set; with Tlast set only each chunk's last prefix is written, to
// (Tlast, Slast)[c].  Arrays [chunk][H][D][D].
struct ScanChunks {
  int m, P;
  const float *Tc, *Sc;
  float *Tlast, *Slast;
};

// CHUNK: the scan chunk fields of Pipe32Args are read (the two-level scan's launches); without it
// the kernel is the plain composition or scan, compiled without them.
template <bool CHUNK>
__global__ void __launch_bounds__(NTH, 1) compose_pipe32_kernel(Pipe32Args a, ScanChunks q) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar_b[2];  // the B pieces of the step with this parity are written
  __shared__ uint64_t bar_f[2];  // the products of the step with this parity are done
  __shared__ uint64_t bar_e[2];  // MMA commits: output half 0 done, all done
  __shared__ uint64_t bar_a[2];  // epilogue of half h done (its A pieces written)
  __shared__ uint32_t tmem_slot;
  __shared__ volatile int abort_flag;
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(sm);
  const int tid = threadIdx.x, warp = tid >> 5;
  const int H = a.H;
  int b, h, ck = 0, s0 = 0, n = a.n;  // n: the steps of this block's chain, from pool row s0
  bool isT = false;  // scan: the T half (starts at I, no addend)
  if (a.scan) {
    isT = (blockIdx.x & 1) == 0;
    b = 0;
    if (CHUNK) {
      h = (blockIdx.x >> 1) % H;
      ck = (blockIdx.x >> 1) / H;
      s0 = ck * q.m;
      n = a.n - s0 < q.m ? a.n - s0 : q.m;
      if (n < 0) n = 0;
    } else {
      h = blockIdx.x >> 1;
    }
  } else {
    b = blockIdx.x % a.B;
    h = blockIdx.x / a.B;
  }
  const bool addend = !isT;
  const float *carry =
      (CHUNK && a.scan && q.Tc && ck > 0) ? (isT ? q.Tc : q.Sc) + ((size_t)(ck - 1) * H + h) * D * D : nullptr;

  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar_b[i], NE);
      mbar_init(&bar_f[i], 1);
      mbar_init(&bar_e[i], 1);
      mbar_init(&bar_a[i], NE / 2);
    }
    mbar_fence_init();
    abort_flag = 0;
  }
  if (warp == 0) {
    tmem_alloc(&tmem_slot, TM_COLS);
    tmem_relinquish();
  }
  const size_t base_bh = ((size_t)b * H + h) * D * D;
  const int j = tid & (D - 1), half = (tid >> 7) & 1, i0 = half * R;
  const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
  float x[R];
  if (tid < NE) {
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int i = i0 + r;
      if (carry) x[r] = carry[(size_t)i * D + j];
      else if (a.scan) x[r] = (isT && i == j) ? 1.f : 0.f;
      else x[r] = a.S_init ? a.S_init[base_bh + (size_t)i * D + j] : 0.f;
    }
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;

  auto entry = [&](int s) -> int64_t {
    int64_t p = a.idx ? (int64_t)a.idx[(size_t)b * a.n + s] : (int64_t)(s0 + s);
    if (p < 0 || p >= a.pool_size) {
      set_error(a.err, HYPIC_EDEVICE);
      p = 0;
    }
    return p;
  };

  if (warp == NE / 32) {
    // ---- control warp: lane 0 issues every MMA ------------------------------------------------
    if ((tid & 31) == 0) {
      tc_fence_after();
      int commits = 0;
      const uint32_t id128 = idesc_f32acc(1, 1, 0, 0, 128, 128), id64 = idesc_f32acc(1, 1, 0, 0, 128, 64);
      bool pending = false;
      for (int s = 0; s < n; ++s) {
        const int bb = s & 1;
        const uint32_t pp = (uint32_t)(s - 1) & 1u;
        const uint32_t dt = tmem + TM_D + (uint32_t)bb * 128;
        const uint32_t ac[3] = {tmem + TM_HI + (uint32_t)bb * 64, tmem + TM_MID, tmem + TM_LO};
        const uint32_t bt = sb + (uint32_t)bb * BUF_B;
        bool ok = mbar_wait_cycles(&bar_b[bb], (uint32_t)(s >> 1) & 1u, a.err);
        if (ok && s > 0) ok = mbar_wait_cycles(&bar_a[0], pp, a.err);
        if (!ok || abort_flag) {
          abort_flag = 1;
          break;
        }
        tc_fence_after();
        // the five smaller terms (A piece pa, B piece pb), smallest first
        const int pa[5] = {2, 1, 0, 1, 0}, pb[5] = {0, 1, 2, 0, 1};
#pragma unroll 1
        for (int kh = 0; kh < 2; ++kh) {
          if (kh == 1) {
            if (s > 0 && !mbar_wait_cycles(&bar_a[1], pp, a.err)) {
              abort_flag = 1;
              break;
            }
            tc_fence_after();
          }
#pragma unroll
          for (int t = 0; t < 5; ++t) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_f16_tmem_a(dt, ac[pa[t]] + kh * 32 + kk * 8,
                             sdesc_sw128(bt + pb[t] * 32768 + kh * 16384 + kk * 32, 16, 1024), id128,
                             (kh | t | kk) != 0);
          }
          pending = true;
        }
        if (abort_flag) break;
        // hi.hi by output half
#pragma unroll
        for (int nh = 0; nh < 2; ++nh) {
#pragma unroll
          for (int kh = 0; kh < 2; ++kh) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_f16_tmem_a(dt + nh * 64, ac[0] + kh * 32 + kk * 8,
                             sdesc_sw128(bt + kh * 16384 + nh * 8192 + kk * 32, 16, 1024), id64, 1u);
          }
          mma_commit(&bar_e[nh]);
        }
        mma_commit(&bar_f[bb]);
        pending = false;
        ++commits;
      }
      if (pending) {
        mma_commit(&bar_e[1]);
        ++commits;
      }
      if (commits > 0) mbar_wait_cycles(&bar_e[1], (uint32_t)(commits - 1) & 1u, nullptr, 200000000LL);
    }
  } else {
    // ---- epilogue and split threads -------------------------------------------------------------
    // This thread's rows i0 .. i0 + 63 of column j as A pieces (contraction half `half`) of the
    // step with parity p.
    auto write_pieces = [&](uint32_t p) {
#pragma unroll
      for (int c0 = 0; c0 < R; c0 += 16) {
        uint32_t p0[8], p1[8], p2[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) split3(x[c0 + 2 * q], x[c0 + 2 * q + 1], p0[q], p1[q], p2[q]);
        const uint32_t col = tmem + lane_base + (uint32_t)(i0 + c0) / 2;
        st8(col + TM_HI + p * 64, p0);
        st8(col + TM_MID, p1);
        st8(col + TM_LO, p2);
      }
      tmem_st_wait();
    };
    // T of step s as three B pieces in buffer s & 1 (K-major [128 i][64 k] blocks, 128-byte
    // swizzle): warp w, rows w + 8 r; lane l, columns 4l .. 4l + 3.
    auto split_T = [&](int s) {
      const float *Tg = a.pool_T + ((size_t)entry(s) * H + h) * D * D;
      uint8_t *bt = sm + (size_t)(s & 1) * BUF_B;
      const int l = tid & 31;
      const uint32_t kb = (uint32_t)l >> 4, chunk = ((uint32_t)l & 15u) >> 1, sub = ((uint32_t)l & 1u) * 8u;
      float4 v[16];
#pragma unroll
      for (int r = 0; r < 16; ++r) v[r] = reinterpret_cast<const float4 *>(Tg + (size_t)(warp + 8 * r) * D)[l];
#pragma unroll
      for (int r = 0; r < 16; ++r) {
        uint32_t p0a, p1a, p2a, p0b, p1b, p2b;
        split3(v[r].x, v[r].y, p0a, p1a, p2a);
        split3(v[r].z, v[r].w, p0b, p1b, p2b);
        const uint32_t off = kb * 16384u + sw128_offset((uint32_t)(warp + 8 * r), chunk) + sub;
        *reinterpret_cast<uint2 *>(bt + off) = make_uint2(p0a, p0b);
        *reinterpret_cast<uint2 *>(bt + 32768 + off) = make_uint2(p1a, p1b);
        *reinterpret_cast<uint2 *>(bt + 65536 + off) = make_uint2(p2a, p2b);
      }
      fence_proxy_async();  // the pieces are read by the MMAs
    };
    // x = this thread's rows of S_{C|0} of step s (or zero in the T half of a scan)
    auto load_s0 = [&](int s) {
      if (addend) {
        const float *Sg = a.pool_S + ((size_t)entry(s) * H + h) * D * D + (size_t)i0 * D + j;
#pragma unroll
        for (int r = 0; r < R; ++r) x[r] = Sg[(size_t)r * D];
      } else {
#pragma unroll
        for (int r = 0; r < R; ++r) x[r] = 0.f;
      }
    };
    auto wait_warp = [&](uint64_t *bar, uint32_t parity) -> bool {
      int ok = 1;
      if ((tid & 31) == 0) {
        ok = !abort_flag && mbar_wait_cycles(bar, parity, a.err);
        if (!ok) abort_flag = 1;
      }
      return __shfl_sync(0xffffffffu, ok, 0) != 0;
    };
    bool live = true;
    if (n > 0) {
      write_pieces(0);
      split_T(0);
      tc_fence_before();
      mbar_arrive(&bar_b[0]);
      load_s0(0);
    }
    for (int s = 0; s < n && live; ++s) {
      if (s + 1 < n) {
        // the other B buffer was last read by the products of step s - 1
        if (s >= 1 && !wait_warp(&bar_f[(s + 1) & 1], (uint32_t)((s - 1) >> 1) & 1u)) {
          live = false;
          break;
        }
        split_T(s + 1);
        mbar_arrive(&bar_b[(s + 1) & 1]);
      }
      if (!wait_warp(&bar_e[half], (uint32_t)s & 1u)) {
        live = false;
        break;
      }
      tc_fence_after();
      const uint32_t dt = tmem + lane_base + TM_D + (uint32_t)(s & 1) * 128 + i0;
#pragma unroll
      for (int hb = 0; hb < R; hb += 32) {
        float dv[32];
        tmem_ld32(dt + hb, dv);
#pragma unroll
        for (int r = 0; r < 32; ++r) x[hb + r] += dv[r];
      }
      if (a.scan && (!CHUNK || !q.Tlast || s == n - 1)) {
        // (one expression per case: computing the row offset separately measured 2.5% slower)
        float *rec = (CHUNK && q.Tlast)
                         ? (isT ? q.Tlast : q.Slast) + ((size_t)ck * H + h) * D * D + (size_t)i0 * D + j
                         : (isT ? a.T_rec : a.S_rec) + ((size_t)(s0 + s) * H + h) * D * D + (size_t)i0 * D + j;
#pragma unroll
        for (int r = 0; r < R; ++r) rec[(size_t)r * D] = x[r];
      }
      if (s + 1 < n) {
        write_pieces((uint32_t)(s + 1) & 1u);
        tc_fence_before();
        mbar_arrive(&bar_a[half]);
        load_s0(s + 1);
      }
    }
    if (live && !abort_flag && !a.scan) {
      float *out = a.S_out + base_bh;
#pragma unroll
      for (int r = 0; r < R; ++r) out[(size_t)(i0 + r) * D + j] = x[r];
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, TM_COLS);
  }
}

}  // namespace

// Pairs in bf16, no seam window and no scan: the pipelined composition above.
cudaError_t launch_compose_pipe(const CUtensorMap &mT, const CUtensorMap &mS, int H, int B, int n,
                                const int32_t *idx, int64_t pool_size, const float *S_init, float *S_out, int *err,
                                cudaStream_t st) {
  PipeArgs a{};
  a.H = H;
  a.B = B;
  a.n = n;
  a.idx = idx;
  a.pool_size = pool_size;
  a.S_init = S_init;
  a.S_out = S_out;
  a.err = err;
  const long long blocks = (long long)B * H;
  if (blocks <= 0) return cudaSuccess;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  cudaError_t e = cudaFuncSetAttribute(compose_pipe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) return e;
  compose_pipe_kernel<<<(unsigned)blocks, NTH, SMEM_BYTES, st>>>(mT, mS, a);
  return cudaGetLastError();
}

namespace {
template <bool CHUNK>
cudaError_t launch_pipe32(const Pipe32Args &a, const ScanChunks &q, long long blocks, cudaStream_t st) {
  if (blocks <= 0) return cudaSuccess;
  if ((reinterpret_cast<uintptr_t>(a.pool_T) & 15) != 0) return cudaErrorInvalidValue;  // rows read as float4
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  cudaError_t e =
      cudaFuncSetAttribute(compose_pipe32_kernel<CHUNK>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM32);
  if (e != cudaSuccess) return e;
  compose_pipe32_kernel<CHUNK><<<(unsigned)blocks, NTH, SMEM32, st>>>(a, q);
  return cudaGetLastError();
}

// Two-level scan plan for H heads and n pairs: P chunks of m pairs, enough block pairs to fill the
// device once and at least 16 pairs a chunk (P = 1: the plain scan, one chain per head).
void scan_plan(int H, int n, int &P, int &m) {
  P = 1;
  m = n;
  int dev = 0, sms = 0;
  if (H <= 0 || n < 32 || cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    return;
  const int fill = (sms + 2 * H - 1) / (2 * H);
  const int p = fill < n / 16 ? fill : n / 16;
  if (p < 2) return;
  m = (n + p - 1) / p;
  P = (n + m - 1) / m;  // every chunk holds at least one pair
}
}  // namespace

// Pairs in fp32, no seam window: the pipelined composition (one chain per request and head).
cudaError_t launch_compose_pipe32(int H, int B, int n, const int32_t *idx, int64_t pool_size, const float *pool_T,
                                  const float *pool_S, const float *S_init, float *S_out, int *err, cudaStream_t st) {
  Pipe32Args a{};
  a.H = H;
  a.B = B;
  a.n = n;
  a.idx = idx;
  a.pool_size = pool_size;
  a.pool_T = pool_T;
  a.pool_S = pool_S;
  a.S_init = S_init;
  a.S_out = S_out;
  a.err = err;
  return launch_pipe32<false>(a, ScanChunks{}, (long long)B * H, st);
}

// Workspace of the two-level scan (0 when the plan is the plain scan): the chunks' totals and the
// carries into chunks 1 .., T and S, [chunk][H][D][D] fp32.
size_t scan_pipe32_workspace_bytes(int H, int n) {
  int P = 1, m = n;
  scan_plan(H, n, P, m);
  return P < 2 ? 0 : (size_t)(2 * P - 1) * 2 * (size_t)H * D * D * sizeof(float);
}

// Inclusive affine scan over fp32 pairs (T, S [n, H, D, D]) into (Tp, Sp).  With fewer heads than
// fill the device and a workspace of scan_pipe32_workspace_bytes(), a two-level scan: (1) every
// chunk of m pairs is scanned from [I | 0] and only its total kept; (2) the totals are scanned,
// giving the carry into each chunk; (3) every chunk is scanned again from its carry, writing its
// prefixes.  The prefixes are those of the composition rule's associativity; the work is about
// twice the plain scan's, the depth about 2 m + P steps instead of n.  Otherwise the plain scan.
cudaError_t launch_scan_pipe32(int H, int n, const float *T, const float *S, float *Tp, float *Sp, void *ws,
                               size_t ws_bytes, int *err, cudaStream_t st) {
  int P = 1, m = n;
  scan_plan(H, n, P, m);
  const size_t need = P < 2 ? 0 : (size_t)(2 * P - 1) * 2 * (size_t)H * D * D * sizeof(float);
  Pipe32Args a{};
  a.H = H;
  a.B = 1;
  a.n = n;
  a.pool_size = n;
  a.pool_T = T;
  a.pool_S = S;
  a.scan = 1;
  a.err = err;
  if (P < 2 || ws == nullptr || ws_bytes < need || (reinterpret_cast<uintptr_t>(ws) & 15) != 0) {
    a.T_rec = Tp;
    a.S_rec = Sp;
    return launch_pipe32<false>(a, ScanChunks{}, 2LL * H, st);
  }
  const size_t blk = (size_t)H * D * D;
  float *totT = static_cast<float *>(ws), *totS = totT + P * blk;
  float *carT = totS + P * blk, *carS = carT + (P - 1) * blk;
  // (1) chunk totals
  ScanChunks q{};
  q.m = m;
  q.P = P;
  q.Tlast = totT;
  q.Slast = totS;
  cudaError_t e = launch_pipe32<true>(a, q, 2LL * H * P, st);
  if (e != cudaSuccess) return e;
  // (2) carries: the inclusive scan of the first P - 1 totals
  Pipe32Args c = a;
  c.n = P - 1;
  c.pool_size = P;
  c.pool_T = totT;
  c.pool_S = totS;
  c.T_rec = carT;
  c.S_rec = carS;
  if ((e = launch_pipe32<false>(c, ScanChunks{}, 2LL * H, st)) != cudaSuccess) return e;
  // (3) every chunk again, from its carry
  q.Tlast = q.Slast = nullptr;
  q.Tc = carT;
  q.Sc = carS;
  a.T_rec = Tp;
  a.S_rec = Sp;
  return launch_pipe32<true>(a, q, 2LL * H * P, st);
}

}  // namespace hypic
