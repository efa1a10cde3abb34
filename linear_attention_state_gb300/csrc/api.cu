// libhypic C ABI: host-side argument checks, the per-device status word and
// dispatch to the kernels.  Every check here runs before anything is enqueued.
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "common.cuh"

namespace hypic {
namespace {

__device__ int g_status_word;  // first device-side error since the last hypic_stream_status()

constexpr int kMaxDevices = 64;
int *g_status_ptr[kMaxDevices];
std::mutex g_status_mu[kMaxDevices];

// Device address of the status word on the current device.  Looked up with the device current;
// only a successful lookup is kept, so a transient failure is retried on the next call.
cudaError_t status_word(int **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_status_mu[dev]);
  if (!g_status_ptr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_status_word);
    if (e != cudaSuccess) return e;
    g_status_ptr[dev] = static_cast<int *>(p);
  }
  *out = g_status_ptr[dev];
  return cudaSuccess;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool ok_ptr(const void *p) { return p != nullptr && aligned16(p); }
bool ok_opt(const void *p) { return p == nullptr || aligned16(p); }

bool dense_family(int f) { return f == HYPIC_FAM_DELTA || f == HYPIC_FAM_GATED_DELTA || f == HYPIC_FAM_KDA; }

// Shape checks common to every call.  Returns HYPIC_OK or the error.
hypic_status check_shape(const hypic_shape *s) {
  if (!s) return HYPIC_EINVAL;
  if (s->H < 0 || s->d_k <= 0 || s->d_v <= 0) return HYPIC_EINVAL;
  if (s->family < HYPIC_FAM_SCALAR_CONST || s->family > HYPIC_FAM_KDA) return HYPIC_EINVAL;
  if (s->in_dtype != HYPIC_F32 && s->in_dtype != HYPIC_BF16) return HYPIC_EINVAL;
  if (s->d_k != s->d_v) return HYPIC_EUNSUPPORTED;
  const int d = s->d_k;
  if (d != 16 && d != 32 && d != 64 && d != 128) return HYPIC_EUNSUPPORTED;
  return HYPIC_OK;
}

// Gate pointers the family needs (alpha unless DELTA; beta for the delta families).
hypic_status check_gates(const hypic_shape *s, const float *alpha, const float *beta) {
  if (s->family != HYPIC_FAM_DELTA && !ok_ptr(alpha)) return HYPIC_EINVAL;
  if (dense_family(s->family) && !ok_ptr(beta)) return HYPIC_EINVAL;
  return HYPIC_OK;
}

// HYPIC_BUILD_PATH=recurrent selects the token-by-token build even where the
// tensor-core path applies (for comparisons); read at every call.
bool force_recurrent() {
  const char *v = getenv("HYPIC_BUILD_PATH");
  return v && strcmp(v, "recurrent") == 0;
}

hypic_status from_cuda(cudaError_t e) { return e == cudaSuccess ? HYPIC_OK : HYPIC_ECUDA; }

hypic_status build_common(const hypic_shape *sh, int32_t n_seg, const SegMap &seg, const void *k,
                          const void *v, const void *q, const float *alpha, const float *beta,
                          float *T_out, float *S_out, float *o_out, bool tokens, void *ws, size_t ws_bytes,
                          cudaStream_t st) {
  if (n_seg == 0 || sh->H == 0) return HYPIC_OK;
  if (!ok_ptr(T_out) || !ok_ptr(S_out)) return HYPIC_EINVAL;
  if (tokens) {  // token pointers are only read when some body is non-empty
    if (!ok_ptr(k) || !ok_ptr(v) || !ok_opt(o_out) || !ok_opt(q)) return HYPIC_EINVAL;
    if (o_out && !ok_ptr(q)) return HYPIC_EINVAL;
    hypic_status r = check_gates(sh, alpha, beta);
    if (r != HYPIC_OK) return r;
  } else {
    o_out = nullptr;
  }
  const bool tc = tokens && build_tc_supported(sh->d_k, sh->family, sh->in_dtype, o_out != nullptr) &&
                  !force_recurrent();
  const bool dtc = tokens && build_decay_tc_supported(sh->d_k, sh->family, sh->in_dtype, o_out != nullptr) &&
                   !force_recurrent();
  if (tc && (ws_bytes < build_tc_min_workspace(n_seg, seg.max_len, o_out != nullptr) || !ok_ptr(ws)))
    return HYPIC_ENOSPACE;
  const bool ktc = tokens && build_kda_tc_supported(sh->d_k, sh->family, sh->in_dtype, o_out != nullptr) &&
                   !force_recurrent();
  if (ktc && (ws_bytes < build_kda_tc_min_workspace(n_seg, seg.max_len) || !ok_ptr(ws))) return HYPIC_ENOSPACE;
  int *err = nullptr;
  cudaError_t e = status_word(&err);
  if (e != cudaSuccess) return HYPIC_ECUDA;
  RecurrentArgs a{};
  a.H = sh->H;
  a.D = sh->d_k;
  a.fam = sh->family;
  a.n_seg = n_seg;
  a.seg = seg;
  a.src = TokenSrc{k, v, q, alpha, beta, sh->in_dtype};
  a.S_in = nullptr;
  a.S_out = S_out;
  a.T_out = T_out;
  a.o_out = o_out;
  a.err = err;
  if (tc) return from_cuda(launch_build_tc(a, ws, ws_bytes, st));
  if (ktc) return from_cuda(launch_build_kda_tc(a, ws, ws_bytes, st));
  if (dtc) return from_cuda(launch_build_decay_tc(a, st));
  return from_cuda(launch_recurrent(a, st));
}

}  // namespace
}  // namespace hypic

using namespace hypic;

extern "C" {

int32_t hypic_abi_version(void) { return 1; }

int64_t hypic_t_size(const hypic_shape *s) {
  if (check_shape(s) != HYPIC_OK) return 0;
  if (s->family == HYPIC_FAM_SCALAR_CONST || s->family == HYPIC_FAM_SCALAR) return 1;
  if (s->family == HYPIC_FAM_DIAG) return s->d_k;
  return (int64_t)s->d_k * s->d_k;
}

const char *hypic_strerror(hypic_status s) {
  switch (s) {
    case HYPIC_OK: return "ok";
    case HYPIC_EINVAL: return "invalid argument";
    case HYPIC_EUNSUPPORTED: return "unsupported shape or family";
    case HYPIC_ECUDA: return "CUDA runtime error";
    case HYPIC_ETIMEOUT: return "bounded wait inside a kernel ran out";
    case HYPIC_ENOSPACE: return "workspace too small";
    case HYPIC_EDEVICE: return "device-side check failed (index or bound out of range)";
    default: return "unknown status";
  }
}

size_t hypic_build_workspace_bytes(const hypic_shape *sh, int32_t n_seg, int64_t max_len) {
  if (check_shape(sh) != HYPIC_OK || n_seg <= 0 || max_len <= 0) return 0;
  if (build_kda_tc_supported(sh->d_k, sh->family, sh->in_dtype, false))
    return build_kda_tc_workspace_bytes(sh->H, n_seg, max_len);
  if (!build_tc_supported(sh->d_k, sh->family, sh->in_dtype, false)) return 0;
  return build_tc_workspace_bytes(sh->H, n_seg, max_len, false);
}

size_t hypic_build_workspace_bytes_outputs(const hypic_shape *sh, int32_t n_seg, int64_t max_len) {
  if (check_shape(sh) != HYPIC_OK || n_seg <= 0 || max_len <= 0) return 0;
  if (!build_tc_supported(sh->d_k, sh->family, sh->in_dtype, true)) return 0;
  return build_tc_workspace_bytes(sh->H, n_seg, max_len, true);
}

size_t hypic_scan_workspace_bytes(const hypic_shape *sh, int32_t n) {
  if (check_shape(sh) != HYPIC_OK || n <= 0 || sh->d_k != sh->d_v) return 0;
  if (!compose_tc_supported(sh->d_k, sh->family)) return 0;
  return scan_pipe32_workspace_bytes(sh->H, n);
}

hypic_status hypic_segment_build(const hypic_shape *sh, const void *k, const void *v, const void *q,
                                 const float *alpha, const float *beta, int64_t len, float *T_out,
                                 float *S_out, float *o_out, void *ws, size_t ws_bytes,
                                 hypic_stream_t stream) {
  hypic_status r = check_shape(sh);
  if (r != HYPIC_OK) return r;
  if (len < 0) return HYPIC_EINVAL;
  SegMap m{nullptr, 0, 0, len, len, len};
  return build_common(sh, 1, m, k, v, q, alpha, beta, T_out, S_out, o_out, len > 0, ws, ws_bytes,
                      (cudaStream_t)stream);
}

hypic_status hypic_segment_build_batched(const hypic_shape *sh, int32_t n_seg, const int64_t *seg_bounds,
                                         int64_t max_len, int64_t n_tokens, const void *k, const void *v,
                                         const void *q, const float *alpha, const float *beta,
                                         float *T_out, float *S_out, float *o_out, void *ws,
                                         size_t ws_bytes, hypic_stream_t stream) {
  hypic_status r = check_shape(sh);
  if (r != HYPIC_OK) return r;
  if (n_seg < 0 || max_len < 0 || n_tokens < 0) return HYPIC_EINVAL;
  if (n_seg > 0 && !ok_ptr(seg_bounds)) return HYPIC_EINVAL;
  SegMap m{seg_bounds, 0, 0, 0, max_len, n_tokens};
  return build_common(sh, n_seg, m, k, v, q, alpha, beta, T_out, S_out, o_out, n_tokens > 0 && max_len > 0, ws,
                      ws_bytes, (cudaStream_t)stream);
}

hypic_status hypic_segment_build_batched_host(const hypic_shape *sh, int32_t n_seg, const int64_t *seg_bounds_host,
                                              int64_t max_len, int64_t n_tokens, const void *k_host,
                                              const void *v_host, const float *alpha_host, const float *beta_host,
                                              void *k_dev, void *v_dev, float *alpha_dev, float *beta_dev,
                                              int64_t *bounds_dev, float *T_out, float *S_out, void *ws,
                                              size_t ws_bytes, hypic_stream_t stream, hypic_stream_t copy_stream,
                                              void *ready_event) {
  hypic_status r = check_shape(sh);
  if (r != HYPIC_OK) return r;
  if (n_seg < 0 || max_len < 0 || n_tokens < 0) return HYPIC_EINVAL;
  if (n_seg == 0 || sh->H == 0) return HYPIC_OK;
  if (!seg_bounds_host || !ok_ptr(bounds_dev)) return HYPIC_EINVAL;
  const bool tokens = n_tokens > 0 && max_len > 0;
  if (tokens) {
    if (!k_host || !v_host || !ok_ptr(k_dev) || !ok_ptr(v_dev)) return HYPIC_EINVAL;
    if (sh->family != HYPIC_FAM_DELTA && (!alpha_host || !ok_ptr(alpha_dev))) return HYPIC_EINVAL;
    if (dense_family(sh->family) && (!beta_host || !ok_ptr(beta_dev))) return HYPIC_EINVAL;
  }
  // Host-side copy plan: the bodies' token rows, checked against the token axis here (the
  // kernels check them again on the device).
  for (int32_t i = 0; i < n_seg; ++i) {
    const int64_t b = seg_bounds_host[2 * i], e = seg_bounds_host[2 * i + 1];
    if (b < 0 || e < b || e - b > max_len || e > n_tokens) return HYPIC_EINVAL;
  }
  const size_t el = sh->in_dtype == HYPIC_BF16 ? 2 : 4;
  const size_t row_kv = (size_t)sh->H * sh->d_k * el;
  const bool per_channel_alpha = sh->family == HYPIC_FAM_DIAG || sh->family == HYPIC_FAM_KDA;
  const size_t row_a = (size_t)sh->H * (per_channel_alpha ? sh->d_k : 1) * sizeof(float);
  const size_t row_b = (size_t)sh->H * sizeof(float);
  const int64_t tsz = hypic_t_size(sh);
  cudaStream_t st = (cudaStream_t)stream, cp = copy_stream ? (cudaStream_t)copy_stream : st;
  // Groups of consecutive segments holding about an eighth of the body tokens each (at least 7/8
  // of an eighth, so that equal bodies a seam shorter than the rest still form groups of one; at
  // most kMaxGroups groups), so that the last group's build, which no copy hides, stays short.
  int64_t body_total = 0;
  for (int32_t i = 0; i < n_seg; ++i) body_total += seg_bounds_host[2 * i + 1] - seg_bounds_host[2 * i];
  constexpr int kMaxGroups = 16;
  const int64_t target = body_total * 7 / 64 > 1 ? body_total * 7 / 64 : 1;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return HYPIC_ECUDA;
  static std::mutex mu[kMaxDevices];
  static cudaEvent_t ev[kMaxDevices][kMaxGroups + 1];
  static bool ev_ready[kMaxDevices];
  std::lock_guard<std::mutex> lock(mu[dev]);
  if (!ev_ready[dev]) {
    for (int i = 0; i <= kMaxGroups; ++i)
      if (cudaEventCreateWithFlags(&ev[dev][i], cudaEventDisableTiming) != cudaSuccess) return HYPIC_ECUDA;
    ev_ready[dev] = true;
  }
  // The copies may overwrite the device buffers only once nothing reads them any more: after the
  // caller's ready event, or else after all the work already on the compute stream.
  if (ready_event) {
    if (cudaStreamWaitEvent(cp, (cudaEvent_t)ready_event, 0) != cudaSuccess) return HYPIC_ECUDA;
  } else if (cp != st) {
    if (cudaEventRecord(ev[dev][kMaxGroups], st) != cudaSuccess) return HYPIC_ECUDA;
    if (cudaStreamWaitEvent(cp, ev[dev][kMaxGroups], 0) != cudaSuccess) return HYPIC_ECUDA;
  }
  if (cudaMemcpyAsync(bounds_dev, seg_bounds_host, sizeof(int64_t) * 2 * n_seg, cudaMemcpyHostToDevice, cp) !=
      cudaSuccess)
    return HYPIC_ECUDA;
  int32_t g0 = 0;
  int groups = 0;
  while (g0 < n_seg) {
    int32_t g1 = g0 + 1;
    if (groups == kMaxGroups - 1) {
      g1 = n_seg;  // the last group takes the rest
    } else {
      int64_t acc = seg_bounds_host[2 * g0 + 1] - seg_bounds_host[2 * g0];
      while (g1 < n_seg && acc < target) {
        acc += seg_bounds_host[2 * g1 + 1] - seg_bounds_host[2 * g1];
        ++g1;
      }
    }
    // Token rows of the group's bodies, each through the end of its last 64-token chunk: the
    // build reads whole chunks (rows past a body's end enter with zero gates), so those rows
    // must hold the request's own tokens, as they do when the inputs are already on the device.
    int64_t r0 = INT64_MAX, r1 = 0;
    for (int32_t i = g0; i < g1; ++i) {
      const int64_t b = seg_bounds_host[2 * i], e = seg_bounds_host[2 * i + 1];
      if (e > b) {
        const int64_t ep = b + (e - b + 63) / 64 * 64;
        r0 = b < r0 ? b : r0;
        r1 = (ep < n_tokens ? ep : n_tokens) > r1 ? (ep < n_tokens ? ep : n_tokens) : r1;
      }
    }
    if (tokens && r1 > r0) {
      const size_t n = (size_t)(r1 - r0);
      auto h2d = [&](void *dst, const void *src, size_t row) {
        return cudaMemcpyAsync(static_cast<char *>(dst) + r0 * row, static_cast<const char *>(src) + r0 * row,
                               n * row, cudaMemcpyHostToDevice, cp);
      };
      if (h2d(k_dev, k_host, row_kv) != cudaSuccess || h2d(v_dev, v_host, row_kv) != cudaSuccess) return HYPIC_ECUDA;
      if (sh->family != HYPIC_FAM_DELTA && h2d(alpha_dev, alpha_host, row_a) != cudaSuccess) return HYPIC_ECUDA;
      if (dense_family(sh->family) && h2d(beta_dev, beta_host, row_b) != cudaSuccess) return HYPIC_ECUDA;
    }
    if (cp != st) {
      if (cudaEventRecord(ev[dev][groups], cp) != cudaSuccess) return HYPIC_ECUDA;
      if (cudaStreamWaitEvent(st, ev[dev][groups], 0) != cudaSuccess) return HYPIC_ECUDA;
    }
    SegMap m{bounds_dev + 2 * g0, 0, 0, 0, max_len, n_tokens};
    r = build_common(sh, g1 - g0, m, k_dev, v_dev, nullptr, sh->family == HYPIC_FAM_DELTA ? nullptr : alpha_dev,
                     dense_family(sh->family) ? beta_dev : nullptr, T_out + (size_t)g0 * sh->H * tsz,
                     S_out + (size_t)g0 * sh->H * sh->d_k * sh->d_v, nullptr, tokens, ws, ws_bytes, st);
    if (r != HYPIC_OK) return r;
    ++groups;
    g0 = g1;
  }
  return HYPIC_OK;
}

hypic_status hypic_seam_advance(const hypic_shape *sh, int32_t B, float *S_inout, const void *q,
                                const void *k, const void *v, const float *alpha, const float *beta,
                                int32_t w, float *o_out, hypic_stream_t stream) {
  hypic_status r = check_shape(sh);
  if (r != HYPIC_OK) return r;
  if (B < 0 || w < 0) return HYPIC_EINVAL;
  if (B == 0 || sh->H == 0 || w == 0) return HYPIC_OK;
  if (!ok_ptr(S_inout) || !ok_opt(o_out)) return HYPIC_EINVAL;
  if (!ok_ptr(k) || !ok_ptr(v) || (o_out && !ok_ptr(q))) return HYPIC_EINVAL;
  r = check_gates(sh, alpha, beta);
  if (r != HYPIC_OK) return r;
  int *err = nullptr;
  if (status_word(&err) != cudaSuccess) return HYPIC_ECUDA;
  RecurrentArgs a{};
  a.H = sh->H;
  a.D = sh->d_k;
  a.fam = sh->family;
  a.n_seg = B;
  a.seg = SegMap{nullptr, w, 0, w, w, (int64_t)B * w};
  a.src = TokenSrc{k, v, q, alpha, beta, sh->in_dtype};
  a.S_in = S_inout;
  a.S_out = S_inout;
  a.T_out = nullptr;
  a.o_out = o_out;
  a.err = err;
  return from_cuda(launch_recurrent(a, (cudaStream_t)stream));
}

static hypic_status chain_common(const hypic_shape *sh, int32_t B, int32_t n, int32_t w, const int32_t *idx,
                                 int64_t pool_size, const void *pool_T, const void *pool_S, bool pair_bf16,
                                 const void *seam_q, const void *seam_k, const void *seam_v,
                                 const float *seam_alpha, const float *seam_beta, const float *S_init,
                                 float *S_out, float *o_out, cudaStream_t st) {
  hypic_status r = check_shape(sh);
  if (r != HYPIC_OK) return r;
  // bf16 pools: delta families only on the d = 128 tensor-core chain
  if (pair_bf16 && dense_family(sh->family) && sh->d_k != 128) return HYPIC_EUNSUPPORTED;
  if (B < 0 || n < 0 || w < 0 || pool_size < 0) return HYPIC_EINVAL;
  if (B == 0 || sh->H == 0) return HYPIC_OK;
  if (!ok_ptr(S_out) || !ok_opt(S_init) || !ok_opt(o_out)) return HYPIC_EINVAL;
  if (n > 0 && (!ok_ptr(idx) || !ok_ptr(pool_T) || !ok_ptr(pool_S) || pool_size == 0)) return HYPIC_EINVAL;
  const bool seams = w > 0 && n > 1;
  if (seams) {
    if (!ok_ptr(seam_k) || !ok_ptr(seam_v) || (o_out && !ok_ptr(seam_q))) return HYPIC_EINVAL;
    r = check_gates(sh, seam_alpha, seam_beta);
    if (r != HYPIC_OK) return r;
  }
  int *err = nullptr;
  if (status_word(&err) != cudaSuccess) return HYPIC_ECUDA;
  ChainArgs a{};
  a.H = sh->H;
  a.D = sh->d_k;
  a.fam = sh->family;
  a.B = B;
  a.n = n;
  a.w = seams ? w : 0;
  a.idx = idx;
  a.pool_size = pool_size;
  a.pool_T = pool_T;
  a.pool_S = pool_S;
  a.pair_bf16 = pair_bf16 ? 1 : 0;
  a.S_init = S_init;
  a.S_out = S_out;
  a.scan = 0;
  a.seam = TokenSrc{seam_k, seam_v, seam_q, seam_alpha, seam_beta, sh->in_dtype};
  a.o_out = seams ? o_out : nullptr;
  a.err = err;
  return from_cuda(launch_chain(a, st));
}

hypic_status hypic_compose(const hypic_shape *sh, int32_t B, int32_t n, const int32_t *idx, int64_t pool_size,
                           const float *pool_T, const float *pool_S, const float *S_init, float *S_out,
                           hypic_stream_t stream) {
  return chain_common(sh, B, n, 0, idx, pool_size, pool_T, pool_S, false, nullptr, nullptr, nullptr, nullptr,
                      nullptr, S_init, S_out, nullptr, (cudaStream_t)stream);
}

hypic_status hypic_compose_bf16(const hypic_shape *sh, int32_t B, int32_t n, const int32_t *idx,
                                int64_t pool_size, const void *pool_T, const void *pool_S, const float *S_init,
                                float *S_out, hypic_stream_t stream) {
  return chain_common(sh, B, n, 0, idx, pool_size, pool_T, pool_S, true, nullptr, nullptr, nullptr, nullptr,
                      nullptr, S_init, S_out, nullptr, (cudaStream_t)stream);
}

hypic_status hypic_assemble(const hypic_shape *sh, int32_t B, int32_t n, int32_t w, const int32_t *idx,
                            int64_t pool_size, const float *pool_T, const float *pool_S, const void *seam_q,
                            const void *seam_k, const void *seam_v, const float *seam_alpha,
                            const float *seam_beta, const float *S_init, float *S_out, float *o_out,
                            hypic_stream_t stream) {
  return chain_common(sh, B, n, w, idx, pool_size, pool_T, pool_S, false, seam_q, seam_k, seam_v, seam_alpha,
                      seam_beta, S_init, S_out, o_out, (cudaStream_t)stream);
}

hypic_status hypic_assemble_bf16(const hypic_shape *sh, int32_t B, int32_t n, int32_t w, const int32_t *idx,
                                 int64_t pool_size, const void *pool_T, const void *pool_S, const void *seam_q,
                                 const void *seam_k, const void *seam_v, const float *seam_alpha,
                                 const float *seam_beta, const float *S_init, float *S_out, float *o_out,
                                 hypic_stream_t stream) {
  return chain_common(sh, B, n, w, idx, pool_size, pool_T, pool_S, true, seam_q, seam_k, seam_v, seam_alpha,
                      seam_beta, S_init, S_out, o_out, (cudaStream_t)stream);
}

hypic_status hypic_pairs_to_bf16(const hypic_shape *sh, int64_t n_pairs, const float *T, const float *S,
                                 void *T_lp, void *S_lp, hypic_stream_t stream) {
  hypic_status r = check_shape(sh);
  if (r != HYPIC_OK) return r;
  if (n_pairs < 0) return HYPIC_EINVAL;
  if (n_pairs == 0 || sh->H == 0) return HYPIC_OK;
  if (!ok_ptr(T) || !ok_ptr(S) || !ok_ptr(T_lp) || !ok_ptr(S_lp)) return HYPIC_EINVAL;
  const int64_t t_elems = n_pairs * sh->H * hypic_t_size(sh);
  const int64_t s_elems = n_pairs * sh->H * (int64_t)sh->d_k * sh->d_v;
  return from_cuda(launch_pairs_to_bf16(T, S, T_lp, S_lp, t_elems, s_elems, (cudaStream_t)stream));
}

hypic_status hypic_affine_scan(const hypic_shape *sh, int32_t n, const float *T, const float *S,
                               float *T_prefix, float *S_prefix, void *ws, size_t ws_bytes,
                               hypic_stream_t stream) {
  hypic_status r = check_shape(sh);
  if (r != HYPIC_OK) return r;
  if (n < 0) return HYPIC_EINVAL;
  if (n == 0 || sh->H == 0) return HYPIC_OK;
  if (!ok_ptr(T) || !ok_ptr(S) || !ok_ptr(T_prefix) || !ok_ptr(S_prefix)) return HYPIC_EINVAL;
  int *err = nullptr;
  if (status_word(&err) != cudaSuccess) return HYPIC_ECUDA;
  ChainArgs a{};
  a.H = sh->H;
  a.D = sh->d_k;
  a.fam = sh->family;
  a.B = 1;
  a.n = n;
  a.w = 0;
  a.idx = nullptr;
  a.pool_size = n;
  a.pool_T = T;
  a.pool_S = S;
  a.pair_bf16 = 0;
  a.S_init = nullptr;
  a.S_out = nullptr;
  a.scan = 1;
  a.T_rec = T_prefix;
  a.S_rec = S_prefix;
  a.seam = TokenSrc{nullptr, nullptr, nullptr, nullptr, nullptr, sh->in_dtype};
  a.o_out = nullptr;
  a.err = err;
  a.ws = ws;
  a.ws_bytes = ws_bytes;
  return from_cuda(launch_chain(a, (cudaStream_t)stream));
}

static bool ok_dtype(hypic_dtype d) { return d == HYPIC_F32 || d == HYPIC_BF16; }
static bool ok_rope(int32_t d, int32_t r, double base) {
  return d >= 2 && d <= 512 && r >= 2 && r <= d && (r % 2) == 0 && base > 1.0 && base < 1e300;
}

hypic_status hypic_rope_shift(int64_t n_rows, int32_t d, int32_t rot_dim, double base, int64_t delta,
                              hypic_dtype dtype, const void *K_in, void *K_out, hypic_stream_t stream) {
  if (n_rows < 0 || !ok_rope(d, rot_dim, base) || !ok_dtype(dtype)) return HYPIC_EINVAL;
  if (n_rows == 0) return HYPIC_OK;
  if (!ok_ptr(K_in) || !ok_ptr(K_out)) return HYPIC_EINVAL;
  int *err = nullptr;
  if (status_word(&err) != cudaSuccess) return HYPIC_ECUDA;
  return from_cuda(launch_rope_shift(K_in, K_out, n_rows, d, rot_dim, base, (long long)delta, dtype, err,
                                     (cudaStream_t)stream));
}

hypic_status hypic_state_rerotate(const hypic_shape *sh, int64_t n, float *S_inout, int32_t rot_dim, double base,
                                  int64_t delta, hypic_stream_t stream) {
  hypic_status r = check_shape(sh);
  if (r != HYPIC_OK) return r;
  if (sh->family != HYPIC_FAM_SCALAR_CONST && sh->family != HYPIC_FAM_SCALAR) return HYPIC_EUNSUPPORTED;
  if (n < 0 || !ok_rope(sh->d_k, rot_dim, base)) return HYPIC_EINVAL;
  if (n == 0 || sh->H == 0) return HYPIC_OK;
  if (!ok_ptr(S_inout)) return HYPIC_EINVAL;
  int *err = nullptr;
  if (status_word(&err) != cudaSuccess) return HYPIC_ECUDA;
  return from_cuda(launch_state_rerotate(S_inout, n * sh->H, sh->d_k, sh->d_v, rot_dim, base, (long long)delta, err,
                                         (cudaStream_t)stream));
}

hypic_status hypic_conv_tail(int32_t C, int32_t k, int32_t n_seg, const int64_t *seg_bounds, int64_t n_tokens,
                             hypic_dtype dtype, const void *x, void *tail_out, hypic_stream_t stream) {
  if (C < 0 || k < 1 || k > 64 || n_seg < 0 || n_tokens < 0 || !ok_dtype(dtype)) return HYPIC_EINVAL;
  if (n_seg == 0 || C == 0 || k == 1) return HYPIC_OK;
  if (!ok_ptr(seg_bounds) || !ok_ptr(tail_out) || (n_tokens > 0 && !ok_ptr(x))) return HYPIC_EINVAL;
  int *err = nullptr;
  if (status_word(&err) != cudaSuccess) return HYPIC_ECUDA;
  return from_cuda(launch_conv_tail(x, n_tokens, C, k, n_seg, seg_bounds, tail_out, dtype, err, (cudaStream_t)stream));
}

hypic_status hypic_conv_seam(int32_t B, int32_t w, int32_t C, int32_t k, hypic_dtype dtype, const void *x_seam,
                             const void *tail, const float *weight, const float *bias, int32_t act, float *y_out,
                             hypic_stream_t stream) {
  if (B < 0 || w < 0 || C < 0 || k < 1 || k > 64 || !ok_dtype(dtype)) return HYPIC_EINVAL;
  if (act != HYPIC_ACT_IDENTITY && act != HYPIC_ACT_SILU) return HYPIC_EINVAL;
  if (B == 0 || w == 0 || C == 0) return HYPIC_OK;
  if (!ok_ptr(x_seam) || !ok_ptr(weight) || !ok_opt(bias) || !ok_ptr(y_out)) return HYPIC_EINVAL;
  if (k > 1 && !ok_ptr(tail)) return HYPIC_EINVAL;
  return from_cuda(launch_conv_seam(x_seam, tail, weight, bias, B, w, C, k, act, dtype, y_out, (cudaStream_t)stream));
}

hypic_status hypic_selftest_bounded_wait(int64_t limit_cycles, hypic_stream_t stream) {
  if (limit_cycles < 0 || limit_cycles > 4000000000LL) return HYPIC_EINVAL;
  int *err = nullptr;
  if (status_word(&err) != cudaSuccess) return HYPIC_ECUDA;
  return from_cuda(launch_bounded_wait_selftest(limit_cycles, err, (cudaStream_t)stream));
}

hypic_status hypic_stream_status(hypic_stream_t stream) {
  cudaStream_t st = (cudaStream_t)stream;
  if (cudaStreamSynchronize(st) != cudaSuccess) return HYPIC_ECUDA;
  int *err = nullptr;
  if (status_word(&err) != cudaSuccess) return HYPIC_ECUDA;
  int host = 0;
  if (cudaMemcpyAsync(&host, err, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess) return HYPIC_ECUDA;
  if (cudaMemsetAsync(err, 0, sizeof(int), st) != cudaSuccess) return HYPIC_ECUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return HYPIC_ECUDA;
  return (hypic_status)host;
}

}  // extern "C"
