// The C ABI declared in include/qmoe.h: host-side validation, workspace
// layout and kernel launches.  Every check runs before the first launch; an
// invalid call launches nothing.
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include "qmoe_common.cuh"

namespace qmoe {

static thread_local char g_err[256] = "";

void set_error(const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof g_err, fmt, ap);
  va_end(ap);
}

int current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
  return dev;
}

int num_sms() {
  static std::atomic<int> cache[kMaxDevices];
  const int dev = current_device();
  if (dev < 0) return 132;
  int n = cache[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 132;
    cache[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

static cudaEvent_t *g_stage_events = nullptr;
static int g_stage_nevents = 0;

void stage_event(int i, cudaStream_t s) {
  if (g_stage_events && i < g_stage_nevents) cudaEventRecord(g_stage_events[i], s);
}

static inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

#define QMOE_REQUIRE(cond, status, ...) \
  do {                                  \
    if (!(cond)) {                      \
      set_error(__VA_ARGS__);           \
      return status;                    \
    }                                   \
  } while (0)

static qmoe_status cuda_status(cudaError_t err, const char *what) {
  if (err == cudaSuccess) return QMOE_OK;
  set_error("%s: %s", what, cudaGetErrorString(err));
  return QMOE_ERR_CUDA;
}

// Bump allocator over the caller's workspace (256-byte aligned regions).
struct Carve {
  char *base;
  size_t off = 0;
  explicit Carve(void *b) : base(static_cast<char *>(b)) {}
  template <typename T>
  T *take(size_t count) {
    off = (off + 255) & ~(size_t)255;
    T *p = base ? reinterpret_cast<T *>(base + off) : nullptr;
    off += count * sizeof(T);
    return p;
  }
};

static qmoe_status check_route_args(const float *logits, int T, int E, int k) {
  QMOE_REQUIRE(logits, QMOE_ERR_INVALID_ARG, "logits is NULL");
  QMOE_REQUIRE(T >= 1, QMOE_ERR_INVALID_ARG, "T must be >= 1 (got %d)", T);
  QMOE_REQUIRE(E >= 1, QMOE_ERR_INVALID_ARG, "E must be >= 1 (got %d)", E);
  QMOE_REQUIRE(k >= 1 && k <= E, QMOE_ERR_INVALID_ARG, "k must be in [1, E] (got k=%d, E=%d)", k, E);
  QMOE_REQUIRE(k <= kMaxTopK, QMOE_ERR_INVALID_ARG, "k must be <= %d (got %d)", kMaxTopK, k);
  QMOE_REQUIRE(E <= kMaxExperts, QMOE_ERR_UNSUPPORTED, "E must be <= %d (got %d)", kMaxExperts, E);
  QMOE_REQUIRE(((uintptr_t)logits & 3u) == 0, QMOE_ERR_MISALIGNED, "logits must be 4-byte aligned");
  QMOE_REQUIRE((long long)T * k <= (1ll << 30), QMOE_ERR_UNSUPPORTED, "T*k too large");
  return QMOE_OK;
}

}  // namespace qmoe

using namespace qmoe;

extern "C" const char *qmoe_last_error(void) { return g_err; }

extern "C" int qmoe_set_stage_events(cudaEvent_t *events, int n_events) {
  g_stage_events = events;
  g_stage_nevents = events ? n_events : 0;
  return 1;
}

extern "C" qmoe_status qmoe_route_topk(const float *logits, const float *router_weights, int T, int E, int k,
                                       int normalize, int32_t *topk_ids,
                                       float *topk_weights, int32_t *expert_offsets, int32_t *perm_to_expanded,
                                       int32_t *expanded_to_perm, void *workspace, size_t *workspace_bytes,
                                       cudaStream_t stream) {
  g_err[0] = 0;
  qmoe_status st = check_route_args(logits, T, E, k);
  if (st != QMOE_OK) return st;
  QMOE_REQUIRE(workspace_bytes, QMOE_ERR_INVALID_ARG, "workspace_bytes is NULL");
  // Routing needs no scratch memory: a call with every output NULL is a size query.
  if (!workspace) *workspace_bytes = 0;
  if (!topk_ids && !topk_weights && !expert_offsets && !perm_to_expanded && !expanded_to_perm) return QMOE_OK;
  QMOE_REQUIRE(topk_ids && topk_weights && expert_offsets && perm_to_expanded && expanded_to_perm,
               QMOE_ERR_INVALID_ARG, "an output pointer is NULL");
  QMOE_REQUIRE(((uintptr_t)router_weights & 3u) == 0, QMOE_ERR_MISALIGNED, "router_weights must be 4-byte aligned");
  RouteOut o{};
  o.mix = router_weights;
  o.ids = topk_ids;
  o.weights = topk_weights;
  o.offsets = expert_offsets;
  o.p2e = perm_to_expanded;
  o.e2p = expanded_to_perm;
  return cuda_status(launch_route(logits, T, E, k, normalize, o, stream), "route launch");
}

extern "C" qmoe_status qmoe_fp4_dequant(const uint8_t *packed, const uint8_t *block_scales,
                                        const float *global_scale, int E, int N, int K, qmoe_fp4_format fmt,
                                        uint16_t *out, cudaStream_t stream) {
  g_err[0] = 0;
  QMOE_REQUIRE(packed && block_scales && out, QMOE_ERR_INVALID_ARG, "packed, block_scales and out must be non-NULL");
  QMOE_REQUIRE((fmt & QMOE_SCALES_KMAJOR) == 0, QMOE_ERR_UNSUPPORTED,
               "dequant takes block scales in the [E, N, K/bs] layout (no QMOE_SCALES_KMAJOR)");
  QMOE_REQUIRE(fmt == QMOE_NVFP4 || fmt == QMOE_MXFP4, QMOE_ERR_UNSUPPORTED, "unknown format %d", (int)fmt);
  QMOE_REQUIRE(E >= 1 && N >= 1 && K >= 1, QMOE_ERR_INVALID_ARG, "E, N, K must be >= 1 (got %d, %d, %d)", E, N, K);
  QMOE_REQUIRE(N % 64 == 0 && K % 64 == 0, QMOE_ERR_UNSUPPORTED, "N and K must be multiples of 64 (got %d, %d)", N,
               K);
  QMOE_REQUIRE(aligned16(packed) && aligned16(block_scales) && aligned16(out) &&
                   (global_scale == nullptr || ((uintptr_t)global_scale & 3u) == 0),
               QMOE_ERR_MISALIGNED, "packed, block_scales and out must be 16-byte aligned");
  return cuda_status(launch_dequant(packed, block_scales, global_scale, E, N, K, (int)fmt, out, stream),
                     "dequant launch");
}

extern "C" qmoe_status qmoe_fp4_scales_kmajor(const uint8_t *block_scales, int E, int N, int K, qmoe_fp4_format fmt,
                                              uint8_t *out, cudaStream_t stream) {
  g_err[0] = 0;
  QMOE_REQUIRE(block_scales && out, QMOE_ERR_INVALID_ARG, "block_scales and out must be non-NULL");
  QMOE_REQUIRE(fmt == QMOE_NVFP4 || fmt == QMOE_MXFP4, QMOE_ERR_UNSUPPORTED, "unknown format %d", (int)fmt);
  QMOE_REQUIRE(E >= 1 && N >= 1 && K >= 1, QMOE_ERR_INVALID_ARG, "E, N, K must be >= 1 (got %d, %d, %d)", E, N, K);
  QMOE_REQUIRE(N % 64 == 0 && K % 64 == 0, QMOE_ERR_UNSUPPORTED, "N and K must be multiples of 64 (got %d, %d)", N,
               K);
  QMOE_REQUIRE(aligned16(block_scales) && aligned16(out), QMOE_ERR_MISALIGNED,
               "block_scales and out must be 16-byte aligned");
  const size_t bytes = (size_t)E * N * (K / block_size((int)fmt));
  const uintptr_t a = (uintptr_t)block_scales, b = (uintptr_t)out;
  QMOE_REQUIRE(a + bytes <= b || b + bytes <= a, QMOE_ERR_INVALID_ARG, "out overlaps block_scales");
  return cuda_status(launch_transpose_bytes(block_scales, E, N, K / block_size((int)fmt), out, stream),
                     "scales_kmajor launch");
}

namespace qmoe {

struct DecodeLayout {
  int32_t *meta;
  float *p1, *p2;
  size_t bytes;
};

// The decode kernel routes in shared memory, so its workspace is the header
// and the FC1 / FC2 partial sums.
static DecodeLayout decode_layout(void *ws, size_t p1_floats, size_t p2_floats) {
  Carve c(ws);
  DecodeLayout L{};
  // [0] unused, [1] device error flag, [2], [3] grid barriers, [4] CTAs out
  L.meta = c.take<int32_t>(QMOE_WORKSPACE_HEADER_BYTES / sizeof(int32_t));
  L.p1 = c.take<float>(p1_floats);
  L.p2 = c.take<float>(p2_floats);
  L.bytes = (c.off + 255) & ~(size_t)255;
  return L;
}

}  // namespace qmoe

namespace qmoe {

// Prefill workspace: routing results, the dequantised weights (unless the
// caller passes them), page-layout scales reconstituted from k-major ones
// (only then), FC1 activations and FC2 rows in permuted order.
struct PrefillLayout {
  int32_t *meta;  // the header: word 1 is the device error flag (the counters are never written here)
  int32_t *ids, *offsets, *p2e, *e2p;
  float *weights, *y;
  uint16_t *xp, *act;
  uint8_t *s1k, *s2k;  // block scales rewritten k-major for the fused GEMMs (scales given as stored)
  size_t bytes;
};

// fused1 / fused2: the FC runs the fused W4A16 GEMM (no dequantised weights
// given); with scales as stored ([E, N, K/bs]) its scales are rewritten
// k-major into the workspace first.
static PrefillLayout prefill_layout(void *ws, int T, int H, int I, int E, int k, int bs, bool fused1, bool fused2,
                                    bool kmajor) {
  const size_t R = (size_t)T * k;
  Carve c(ws);
  PrefillLayout L{};
  L.meta = c.take<int32_t>(QMOE_WORKSPACE_HEADER_BYTES / sizeof(int32_t));
  L.ids = c.take<int32_t>(R);
  L.weights = c.take<float>(R);
  L.offsets = c.take<int32_t>((size_t)E + 1);
  L.p2e = c.take<int32_t>(R);
  L.e2p = c.take<int32_t>(R);
  L.act = c.take<uint16_t>(R * I);
  L.y = c.take<float>(R * H);
  if (fused1) L.xp = c.take<uint16_t>(R * H);
  if (fused1 && !kmajor) L.s1k = c.take<uint8_t>((size_t)E * 2 * I * (H / bs));
  if (fused2 && !kmajor) L.s2k = c.take<uint8_t>((size_t)E * H * (I / bs));
  L.bytes = (c.off + 255) & ~(size_t)255;
  return L;
}

// T * k > QMOE_GEMV_MAX_ROWS: route, grouped GEMMs (fused W4A16, or bf16 over
// dequantised weights the caller gives), weighted un-permute.  Arguments
// already checked by the caller: routing sizes, format, H and I,
// swiglu_fusion, alpha / beta / limit.
static qmoe_status prefill_forward(const uint16_t *x, const float *logits, const float *mix, const uint8_t *fc1_w,
                                   const uint8_t *fc1_s,
                                   const float *fc1_g, const uint8_t *fc2_w, const uint8_t *fc2_s, const float *fc2_g,
                                   const uint16_t *fc1_wd, const uint16_t *fc2_wd, int fmt, bool kmajor, int T, int H,
                                   int I, int E, int k, int normalize, int fusion, float alpha, float beta,
                                   float limit, uint16_t *out, int32_t *topk_ids_out, void *workspace,
                                   size_t *workspace_bytes, cudaStream_t stream) {
  QMOE_REQUIRE((long long)T * k <= (1LL << 30), QMOE_ERR_UNSUPPORTED, "T*k too large");
  const int bs = block_size(fmt);
  const bool need_w1 = fc1_wd == nullptr, need_w2 = fc2_wd == nullptr;
  const PrefillLayout need = prefill_layout(nullptr, T, H, I, E, k, bs, need_w1, need_w2, kmajor);
  if (!workspace) {
    *workspace_bytes = need.bytes;
    return QMOE_OK;
  }
  QMOE_REQUIRE(*workspace_bytes >= need.bytes, QMOE_ERR_WORKSPACE, "workspace too small: %zu < %zu bytes",
               *workspace_bytes, need.bytes);
  QMOE_REQUIRE(x && out, QMOE_ERR_INVALID_ARG, "x and out must be non-NULL");
  QMOE_REQUIRE((!need_w1 || (fc1_w && fc1_s)) && (!need_w2 || (fc2_w && fc2_s)), QMOE_ERR_INVALID_ARG,
               "weights and scales must be non-NULL when no dequantised weights are given");
  QMOE_REQUIRE(aligned16(x) && aligned16(out) && aligned16(workspace) && (!fc1_wd || aligned16(fc1_wd)) &&
                   (!fc2_wd || aligned16(fc2_wd)) && (!need_w1 || (aligned16(fc1_w) && aligned16(fc1_s))) &&
                   (!need_w2 || (aligned16(fc2_w) && aligned16(fc2_s))),
               QMOE_ERR_MISALIGNED, "x, out, workspace, weights and scales must be 16-byte aligned");
  QMOE_REQUIRE((fc1_g == nullptr || ((uintptr_t)fc1_g & 3u) == 0) && (fc2_g == nullptr || ((uintptr_t)fc2_g & 3u) == 0),
               QMOE_ERR_MISALIGNED, "global scales must be 4-byte aligned");
  const PrefillLayout L = prefill_layout(workspace, T, H, I, E, k, bs, need_w1, need_w2, kmajor);
  RouteOut ro{};
  ro.mix = mix;
  ro.ids = topk_ids_out ? topk_ids_out : L.ids;
  ro.weights = L.weights;
  ro.offsets = L.offsets;
  ro.p2e = L.p2e;
  ro.e2p = L.e2p;
  stage_event(0, stream);
  cudaError_t err = launch_route(logits, T, E, k, normalize, ro, stream);
  if (err != cudaSuccess) return cuda_status(err, "route launch");
  stage_event(1, stream);
  // fused FCs read k-major block scales: [E, N, K/bs] -> [E, K/bs, N] when given as stored
  const uint8_t *s1k = fc1_s, *s2k = fc2_s;
  if (need_w1 && !kmajor) {
    err = launch_transpose_bytes(fc1_s, E, 2 * I, H / bs, L.s1k, stream);
    if (err != cudaSuccess) return cuda_status(err, "scale transpose launch");
    s1k = L.s1k;
  }
  if (need_w2 && !kmajor) {
    err = launch_transpose_bytes(fc2_s, E, H, I / bs, L.s2k, stream);
    if (err != cudaSuccess) return cuda_status(err, "scale transpose launch");
    s2k = L.s2k;
  }
  stage_event(2, stream);
  PrefillArgs a{};
  a.fmt = fmt; a.T = T; a.H = H; a.I = I; a.E = E; a.k = k;
  a.alpha = alpha; a.beta = beta; a.limit = limit; a.fusion = fusion;
  a.x = x; a.offsets = L.offsets; a.p2e = L.p2e; a.e2p = L.e2p; a.weights = L.weights;
  a.w1 = fc1_w; a.s1k = s1k; a.g1 = fc1_g; a.w2 = fc2_w; a.s2k = s2k; a.g2 = fc2_g;
  a.w1d = fc1_wd; a.w2d = fc2_wd; a.xp = L.xp; a.act = L.act; a.y = L.y; a.out = out;
  a.err_flag = L.meta + 1;
  return cuda_status(launch_prefill(a, stream), "prefill launch");
}

}  // namespace qmoe

extern "C" qmoe_status qmoe_check_device_error(void *workspace, cudaStream_t stream) {
  g_err[0] = 0;
  void *ws = workspace;
  if (!ws) {  // the static scratch of the no-alloc entry point on this device
    const qmoe_status st = no_alloc_scratch(&ws);
    if (st != QMOE_OK) return st;
  }
  QMOE_REQUIRE(aligned16(ws), QMOE_ERR_MISALIGNED, "workspace must be 16-byte aligned");
  int32_t *flag_dev = static_cast<int32_t *>(ws) + 1;  // header word 1
  int32_t flag = 0;
  cudaError_t err = cudaMemcpyAsync(&flag, flag_dev, sizeof flag, cudaMemcpyDeviceToHost, stream);
  if (err == cudaSuccess) err = cudaStreamSynchronize(stream);
  if (err != cudaSuccess) return cuda_status(err, "reading the device error flag");
  if (flag == 0) return QMOE_OK;
  err = cudaMemsetAsync(flag_dev, 0, sizeof flag, stream);
  if (err == cudaSuccess) err = cudaStreamSynchronize(stream);
  if (err != cudaSuccess) return cuda_status(err, "clearing the device error flag");
  set_error("a bounded wait inside a kernel gave up (device error flag %d): the outputs of the calls on this "
            "workspace since the last check are not to be trusted", (int)flag);
  return QMOE_ERR_DEVICE;
}

extern "C" qmoe_status qmoe_fp4_moe_forward(const uint16_t *x, const float *logits, const float *router_weights,
                                            const uint8_t *fc1_w,
                                            const uint8_t *fc1_s, const float *fc1_g, const uint8_t *fc2_w,
                                            const uint8_t *fc2_s, const float *fc2_g, const uint16_t *fc1_wd,
                                            const uint16_t *fc2_wd, qmoe_fp4_format fmt, int T, int H, int I, int E,
                                            int k, int normalize, int swiglu_fusion, float alpha, float beta,
                                            float limit, uint16_t *out, int32_t *topk_ids_out, void *workspace,
                                            size_t *workspace_bytes, cudaStream_t stream) {
  g_err[0] = 0;
  qmoe_status st = check_route_args(logits, T, E, k);
  if (st != QMOE_OK) return st;
  QMOE_REQUIRE(workspace_bytes, QMOE_ERR_INVALID_ARG, "workspace_bytes is NULL");
  QMOE_REQUIRE(((uintptr_t)router_weights & 3u) == 0, QMOE_ERR_MISALIGNED, "router_weights must be 4-byte aligned");
  const bool kmajor = (fmt & QMOE_SCALES_KMAJOR) != 0;
  const bool primed = (fmt & QMOE_WORKSPACE_PRIMED) != 0;
  const bool multirow = (fmt & QMOE_DECODE_MULTIROW) != 0;
  const int base_fmt = (int)fmt & ~(int)(QMOE_SCALES_KMAJOR | QMOE_WORKSPACE_PRIMED | QMOE_DECODE_MULTIROW);
  QMOE_REQUIRE(!multirow || kmajor, QMOE_ERR_UNSUPPORTED,
               "QMOE_DECODE_MULTIROW needs k-major block scales (QMOE_SCALES_KMAJOR)");
  QMOE_REQUIRE(base_fmt == QMOE_NVFP4 || base_fmt == QMOE_MXFP4, QMOE_ERR_UNSUPPORTED, "unknown format %d", (int)fmt);
  QMOE_REQUIRE(H >= 64 && I >= 64, QMOE_ERR_INVALID_ARG, "H and I must be >= 64 (got %d, %d)", H, I);
  QMOE_REQUIRE(H % 64 == 0 && I % 64 == 0, QMOE_ERR_UNSUPPORTED, "H and I must be multiples of 64 (got %d, %d)", H,
               I);
  QMOE_REQUIRE(swiglu_fusion >= 0 && swiglu_fusion <= 2, QMOE_ERR_UNSUPPORTED,
               "swiglu_fusion must be 0, 1 (interleaved) or 2 (concatenated) (got %d)", swiglu_fusion);
  // 0 is read as 1: the pages' backward-compatibility remap for QMoE
  const int fusion = swiglu_fusion == 2 ? 2 : 1;
  QMOE_REQUIRE(!std::isnan(alpha) && !std::isnan(beta) && !std::isnan(limit), QMOE_ERR_INVALID_ARG,
               "alpha, beta and limit must not be NaN");
  const long long R = (long long)T * k;
  if (R > QMOE_GEMV_MAX_ROWS)
    return prefill_forward(x, logits, router_weights, fc1_w, fc1_s, fc1_g, fc2_w, fc2_s, fc2_g, fc1_wd, fc2_wd, base_fmt, kmajor, T, H,
                           I, E, k, normalize, fusion, alpha, beta, limit, out, topk_ids_out, workspace,
                           workspace_bytes, stream);
  QMOE_REQUIRE(H <= 16384 && I <= 16384, QMOE_ERR_UNSUPPORTED, "decode path needs H, I <= 16384");
  // Scales as stored ([E, N, K/bs]): moe_layer_kernel (layer.cu).  k-major
  // scales: moe_decode_kernel (decode.cu, every row of an expert in one pass)
  // unless one SM's share of the FC1 stream is short (under 16 units, all
  // rows counted once), where moe_layer_kernel's earlier stream start wins;
  // QMOE_DECODE_MULTIROW forces decode.cu.
  LayerPlan plan;
  DkPlan dplan;
  size_t p1_floats = 0, p2_floats = 0;
  bool use_dk = false;
  if (kmajor) {
    st = make_dk_plan(base_fmt, T, H, I, E, k, dplan, p1_floats, p2_floats);
    if (st != QMOE_OK) return st;
    const double units_per_sm = (double)R * dplan.f[0].ct * dplan.f[0].ku / (double)num_sms();
    use_dk = multirow || units_per_sm >= 16.0;
  }
  if (!use_dk) {
    st = make_layer_plan(base_fmt, kmajor, T, H, I, E, k, plan, p1_floats, p2_floats);
    if (st != QMOE_OK) return st;
  }
  const DecodeLayout need = decode_layout(nullptr, p1_floats, p2_floats);
  if (!workspace) {
    *workspace_bytes = need.bytes;
    return QMOE_OK;
  }
  QMOE_REQUIRE(*workspace_bytes >= need.bytes, QMOE_ERR_WORKSPACE, "workspace too small: %zu < %zu bytes",
               *workspace_bytes, need.bytes);
  QMOE_REQUIRE(x && fc1_w && fc1_s && fc2_w && fc2_s && out, QMOE_ERR_INVALID_ARG,
               "x, weights, scales and out must be non-NULL");
  QMOE_REQUIRE(aligned16(x) && aligned16(fc1_w) && aligned16(fc1_s) && aligned16(fc2_w) && aligned16(fc2_s) &&
                   aligned16(out) && aligned16(workspace),
               QMOE_ERR_MISALIGNED, "x, weights, scales, out and workspace must be 16-byte aligned");
  QMOE_REQUIRE((fc1_g == nullptr || ((uintptr_t)fc1_g & 3u) == 0) && (fc2_g == nullptr || ((uintptr_t)fc2_g & 3u) == 0),
               QMOE_ERR_MISALIGNED, "global scales must be 4-byte aligned");

  const DecodeLayout L = decode_layout(workspace, p1_floats, p2_floats);
  LayerArgs g{};
  g.fmt = base_fmt;
  g.T = T; g.H = H; g.I = I; g.E = E; g.k = k;
  g.alpha = alpha; g.beta = beta; g.limit = limit; g.fusion = fusion;
  g.logits = logits; g.mix = router_weights; g.normalize = normalize; g.route_n = route_keys_per_lane(E, k);
  g.ids_out = topk_ids_out;
  g.x = x;
  g.w1 = fc1_w; g.s1 = fc1_s; g.g1 = fc1_g;
  g.w2 = fc2_w; g.s2 = fc2_s; g.g2 = fc2_g;
  g.meta = L.meta;
  g.p1 = L.p1; g.p2 = L.p2; g.out = out;

  stage_event(0, stream);
  // the error flag and the grid-barrier counters start every call at 0: reset
  // here, or (primed workspace) left at 0 by the previous decode kernel
  cudaError_t err = cudaSuccess;
  if (!primed) {
    err = cudaMemsetAsync(L.meta, 0, QMOE_WORKSPACE_HEADER_BYTES, stream);
    if (err != cudaSuccess) return cuda_status(err, "counter reset");
  }
  err = use_dk ? launch_dk(g, dplan, primed, stream) : launch_layer(g, plan, E, primed, stream);
  if (err == cudaErrorCooperativeLaunchTooLarge && g_err[0]) return QMOE_ERR_CUDA;  // message already set
  if (err != cudaSuccess) return cuda_status(err, "layer launch");
  stage_event(1, stream);
  return QMOE_OK;
}
