// Shared device helpers and host-side declarations of the QMoE CUDA library.
// Format decoding follows "MoE and QMoE - CUDA Operator Documentation" §6.5 /
// §9b (E2M1 codes, E4M3FN and E8M0 block scales, fp32 global scale).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/qmoe.h"

namespace qmoe {

constexpr int kNvfp4Block = 16;
constexpr int kMxfp4Block = 32;
constexpr int kMaxExperts = 256;   // warp top-k holds at most 8 keys per lane
constexpr int kMaxTopK = 8;

__host__ __device__ inline int block_size(int fmt) { return fmt == QMOE_NVFP4 ? kNvfp4Block : kMxfp4Block; }

// ---- element codecs (device) -------------------------------------------------

// Two E2M1 codes (low nibble = element 2j, high nibble = element 2j+1) -> f16x2,
// exact, with the sm_100+ hardware converter (no lookup table).
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte_in_low_bits) {
  uint32_t r;
  asm("{ .reg .b8 t; cvt.u8.u32 t, %1; cvt.rn.f16x2.e2m1x2 %0, t; }" : "=r"(r) : "r"(byte_in_low_bits));
  return r;
}

// d = a * b + c with a, b fp16 and c, d fp32; the product is formed exactly.
__device__ __forceinline__ float fma_f16_f32(uint16_t a, uint16_t b, float c) {
  float d;
  asm("fma.rn.f32.f16 %0, %1, %2, %3;" : "=f"(d) : "h"(a), "h"(b), "f"(c));
  return d;
}

// E4M3FN byte -> fp32, exact for every code (subnormals included); S.1111.111 -> NaN.
// The 7 exponent/mantissa bits are placed at the fp32 exponent/mantissa
// position (which gives value * 2^-120, exactly, as an fp32 number, subnormal
// for exponent field 0) and rescaled by 2^120.
__device__ __forceinline__ float e4m3_to_f32(uint32_t b) {
  uint32_t em = b & 0x7Fu;
  float f = __uint_as_float(em << 20) * 0x1p120f;
  if (em == 0x7Fu) f = __uint_as_float(0x7FC00000u);
  return (b & 0x80u) ? -f : f;
}

// E8M0 byte -> fp32: 2^(b-127); 0xFF -> NaN; 0 -> 2^-127 (an fp32 subnormal).
__device__ __forceinline__ float e8m0_to_f32(uint32_t b) {
  b &= 0xFFu;
  if (b == 0xFFu) return __uint_as_float(0x7FC00000u);
  if (b == 0u) return __uint_as_float(0x00400000u);
  return __uint_as_float(b << 23);
}

__device__ __forceinline__ float scale_to_f32(int fmt, uint32_t b) {
  return fmt == QMOE_NVFP4 ? e4m3_to_f32(b) : e8m0_to_f32(b);
}

// fp32 -> bf16 bits, round to nearest even; NaN -> 0x7FC0.
__device__ __forceinline__ uint32_t f32_to_bf16_rne(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7FFFFFFFu) > 0x7F800000u) return 0x7FC0u;
  return (u + 0x7FFFu + ((u >> 16) & 1u)) >> 16;
}

__device__ __forceinline__ float bf16_to_f32(uint32_t bits16) { return __uint_as_float(bits16 << 16); }

// SwiGLU of one (gate, linear) pair ("MoE and QMoE - CUDA Operator
// Documentation" §8): G = min(gate, limit), L = clamp(linear, -limit, limit),
// G * sigmoid(alpha * G) * (L + beta).
__device__ __forceinline__ float swiglu(float gate, float lin, float alpha, float beta, float limit) {
  const float G = fminf(gate, limit);
  const float L = fmaxf(fminf(lin, limit), -limit);
  return G * (1.0f / (1.0f + expf(-alpha * G))) * (L + beta);
}

__device__ __forceinline__ uint32_t lane_id() { return threadIdx.x & 31u; }

// ---- host side -------------------------------------------------------------------

void set_error(const char *fmt, ...);
// Benchmark instrumentation: record stage event i on `s` when the caller set
// events with qmoe_set_stage_events (a no-op otherwise).
void stage_event(int i, cudaStream_t s);
int num_sms();
// Per-device host caches (kernel attributes, symbol addresses) hold this many devices.
constexpr int kMaxDevices = 64;
// The current device, or -1 when there is none or it is outside [0, kMaxDevices).
int current_device();
// Device address of the no-alloc entry point's static scratch on the current
// device (looked up once per device).
qmoe_status no_alloc_scratch(void **addr);

// Routing of few tokens: one CTA does top-k, softmax and the stable expert
// ranking for T <= kFusedRouteMaxTokens tokens.
constexpr int kFusedRouteMaxTokens = 64;

struct RouteOut {
  const float *mix;    // [T, E] router_weights (mixing weights gathered at the selection), or null
  int32_t *ids;        // [T*k]
  float *weights;      // [T*k]
  int32_t *offsets;    // [E+1]
  int32_t *p2e;        // [T*k]
  int32_t *e2p;        // [T*k]
};

cudaError_t launch_route(const float *logits, int T, int E, int k, int normalize, const RouteOut &o,
                         cudaStream_t stream);
// Keys per lane of the warp top-k for E experts and top-k (1, 2, 4 or 8).
int route_keys_per_lane(int E, int k);

// Decode layer (R = T*k <= 64 rows): arguments of the fused kernel.
struct LayerArgs {
  int fmt, T, H, I, E, k;
  float alpha, beta, limit;
  int fusion;              // FC1 gate/linear columns: 1 interleaved (2m, 2m + 1), 2 concatenated (m, I + m)
  const float *logits;     // fp32 [T, E] router logits
  const float *mix;        // fp32 [T, E] router_weights (mixing weights), or null
  int normalize, route_n;  // routing: renormalise over the k; keys per lane (1, 2, 4, 8)
  int32_t *ids_out;        // [T, k] selected experts, or null
  const uint16_t *x;       // bf16 [T, H]
  const uint8_t *w1, *s1, *w2, *s2;
  const float *g1, *g2;
  int32_t *meta;           // workspace header: [1] device error flag, [2], [3] grid barrier counters,
                           // [4] CTAs out; [2..4] are zero at launch and the kernel leaves them zero
  float *p1, *p2;          // fp32 partial sums of FC1 / FC2 (split-K segments)
  uint16_t *out;           // [T, H] bf16
  CUtensorMap tm_s1, tm_s2;  // block scales as 2-D byte arrays (when FcPlan::tma)
  CUtensorMap tm_w1, tm_w2;  // packed weights as 2-D word arrays [E*K rows][N/8 words] (k-major decode, DkFc::ct > 1)
};

constexpr int kCostRows = 64;  // rows of one expert in the decode window (T * k <= 64)

// Geometry of one FC for the decode kernel (host-computed).  Unit = 16*RGS k
// rows x NT columns; thread (w, rg) owns column word w of k-group rg.
struct FcPlan {
  int K, N, NT, ct, NW, RGS;
  int nkg;      // K / 16
  int ku;       // units per (expert, column tile)
  int nblocks;  // K / block size
  int WB;       // scale window, in blocks
  int tma;      // 1: scale windows are 16-block tensor copies (nblocks % 16 == 0)
  int box_rows; // rows of one scale tensor copy
  int rg_stride;  // bytes between row groups in a weight ring slot
  int kn;       // 1: block scales are k-major [E, nblocks, N]; a unit's scale rows ride in its ring slot
  int bpu;      // scale block rows one unit touches (k-major)
  int sc_off;   // offset of those rows in a ring slot
  int pass_cost;  // split: charge of a pass start, in 1/64 of a unit decoded for one row
  int ucost[kCostRows];  // split: cost of one unit of an r-row expert at [r - 1] (same scale)
};
struct LayerPlan {
  FcPlan f[2];
  int ring;  // weight ring slots (3 or 4)
  int slot_bytes, win_bytes;
  int sw_off, st_off, xs_off, xr_off, smem;
};
// Geometry of one FC for the k-major decode kernel (host-computed): unit =
// UK = 16 * RGS k rows x NT columns; consumer thread (w, rg) owns column word
// w (8 columns) of k-group rg of every unit.
struct DkFc {
  int K, N, NT, ct, NW, RGS, lg_rgs, UK;
  int ku;         // units per (expert, column tile)
  int nkg;        // K / 16
  int nblocks;    // K / block size
  int bpu;        // scale block rows one unit touches
  int row_bytes;  // NT / 2
  int rg_stride;  // bytes between row groups in a ring slot
  int sc_off;     // offset of the unit's scale rows in its slot
  int cap;        // partial rows one CTA's region holds
  int u0, u1;     // split cost of a unit of an r-row expert: chunks * u0 + r * u1
};
struct DkPlan {
  DkFc f[2];
  int slot_bytes, win_off, pre_off, smem;  // dynamic shared memory: the ring at 0, windows, FC2 activations
  int pass;                                // split cost of a row chunk's start
};
qmoe_status make_dk_plan(int fmt, int T, int H, int I, int E, int k, DkPlan &P, size_t &p1_floats,
                         size_t &p2_floats);
cudaError_t launch_dk(const LayerArgs &a, const DkPlan &P, bool pdl, cudaStream_t stream);

qmoe_status make_layer_plan(int fmt, bool kmajor, int T, int H, int I, int E, int k, LayerPlan &L,
                            size_t &p1_floats, size_t &p2_floats);
// pdl: launch with programmatic dependent launch (the header is already zero,
// so no memset sits between this kernel and the previous one).
cudaError_t launch_layer(LayerArgs &a, const LayerPlan &L, int E, bool pdl, cudaStream_t stream);

// Programmatic dependent launch: let the next kernel in the stream be scheduled /
// wait here until the previous kernel's results are visible.
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

cudaError_t launch_dequant(const uint8_t *packed, const uint8_t *scales, const float *g, int E, int N, int K,
                           int fmt, uint16_t *out, cudaStream_t stream);
// out[e][c][r] = in[e][r][c] for an [E, rows, cols] byte array (both
// directions of the block-scale layout conversion).
cudaError_t launch_transpose_bytes(const uint8_t *in, int E, int rows, int cols, uint8_t *out, cudaStream_t stream);

// Fused W4A16 grouped GEMM of one FC at prefill (prefill_fp4.cu): packed
// codes [E, K, N/2], k-major block scales [E, K/bs, N], decoded inside the GEMM.
struct Fp4GemmArgs {
  int mode;                 // 0: FC1, gate / linear interleaved; 1: FC1 concatenated; 2: FC2
  int fmt, R, E, H, I;
  const uint8_t *w, *s;     // packed codes, k-major block scales
  const float *gscale;      // [E] or null
  const uint16_t *A;        // bf16 activation rows in expert order: FC1 x gathered [R, H]; FC2 act [R, I]
  const int32_t *offsets;   // [E + 1]
  uint16_t *out_a;          // FC1: act [R, I] bf16
  float *out_y;             // FC2: y [R, H] fp32
  float alpha, beta, limit;
  int32_t *err_flag;
};
cudaError_t launch_fp4_gemm(const Fp4GemmArgs &a, cudaStream_t stream);

// Prefill (T * k > 64): per FC, the fused W4A16 GEMM over the packed weights,
// or the bf16 grouped GEMM over dequantised weights the caller passes.
struct PrefillArgs {
  int fmt, T, H, I, E, k;
  float alpha, beta, limit;
  int fusion;                // FC1 gate/linear columns: 1 interleaved, 2 concatenated
  const uint16_t *x;         // bf16 [T, H]
  const int32_t *offsets;    // [E + 1]
  const int32_t *p2e, *e2p;  // [T * k] permute maps
  const float *weights;      // [T * k] routing weights
  const uint8_t *w1, *s1k;   // FC1 packed codes [E, H, I] bytes and k-major scales [E, H/bs, 2I]
  const uint8_t *w2, *s2k;   // FC2 packed codes [E, I, H/2] and k-major scales [E, I/bs, H]
  const float *g1, *g2;      // global scales [E] or null
  const uint16_t *w1d;       // bf16 [E, 2I, H] given by the caller, or null (fused FC1)
  const uint16_t *w2d;       // bf16 [E, H, I] given by the caller, or null (fused FC2)
  uint16_t *xp;              // bf16 [T * k, H] x gathered in expert order (fused FC1), or null
  uint16_t *act;             // bf16 [T * k, I] FC1 activations, permuted order
  float *y;                  // fp32 [T * k, H] FC2 rows, permuted order
  uint16_t *out;             // bf16 [T, H]
  int32_t *err_flag;         // the workspace's device error flag (header word 1)
};
cudaError_t launch_prefill(const PrefillArgs &a, cudaStream_t stream);

}  // namespace qmoe
