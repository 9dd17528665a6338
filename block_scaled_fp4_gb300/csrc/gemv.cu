// Decode GEMVs of the FP4 MoE layer: FC1 (+ SwiGLU) and FC2 (+ weighted
// un-permute), with the E2M1 weights dequantised in registers.
//
// Prior art on the pages ("[CUDA] Speed up the NVFP4 QMoE decode GEMV and
// enable it for MTP verify", PR #31159; operator doc §9b.2/§9b.3): coalesced
// weight and scale streams, weight loads batched ahead of their decode, a
// table-free E2M1 decode, the block scale applied to a per-block partial sum
// instead of to every weight, fp32 accumulation for bf16 activations, and a
// 64-expanded-row window.  Design here (sm_103a):
//  * one CTA = one active expert x 64 output columns x all of K; 256 threads =
//    8 column words (8 columns each, one 32-bit load per k row) x 32 k-groups;
//    a k-group owns whole scale blocks (16 rows NVFP4, 32 rows MXFP4);
//  * E2M1 pairs decode with the hardware cvt.rn.f16x2.e2m1x2 (one instruction
//    per two weights) and multiply-accumulate with fma.rn.f32.f16 (fp16
//    operands, exact product, fp32 accumulator);
//  * activations are staged in shared memory as fp16 after an exact
//    power-of-two rescale per row (largest |x| in [2^14, 2^15)), so every
//    finite bf16 activation stays in fp16 range; the factor is undone on the
//    fp32 result;
//  * the per-block partial sum is multiplied once by the block scale; NVFP4
//    scales are used as E4M3 * 2^-120 (bits moved into fp32 position, exact)
//    and the 2^120 is folded into the per-expert global scale at the end;
//  * k-group partials are reduced in shared memory in a fixed order
//    (deterministic), then FC1 applies SwiGLU and writes bf16 activations;
//    FC2 writes fp32 rows and the last CTA to finish a column tile (arrival
//    counter, no waiting) forms out[t] = bf16(sum_j w[t][j] * y[t*k+j]) in
//    fixed j order.
#include <cuda_fp16.h>

#include "qmoe_common.cuh"

namespace qmoe {

constexpr int kTileN = 64;          // output columns per CTA
constexpr int kGemvThreads = 256;
constexpr int kWords = kTileN / 8;  // 32-bit words (8 codes) per k row in a tile
constexpr int kKGroups = kGemvThreads / kWords;  // 32
constexpr int kRowChunk = 4;        // rows decoded together

int gemv_fc2_counter_words(int H) { return H / kTileN; }

// Raw block scale as fp32.  NVFP4: E4M3 value * 2^-120 (exact); MXFP4: 2^(b-127).
// `special` is set for codes that need the exact slow path (NaN; E8M0 0 / 255).
template <int FMT>
__device__ __forceinline__ float raw_scale(uint32_t b, bool &special) {
  if (FMT == QMOE_NVFP4) {
    special |= (b & 0x7Fu) == 0x7Fu;
    const float f = __uint_as_float((b & 0x7Fu) << 20);
    return (b & 0x80u) ? -f : f;
  } else {
    special |= (b == 0u) || (b == 0xFFu);
    return __uint_as_float(b << 23);
  }
}
template <int FMT>
__device__ __forceinline__ float exact_raw_scale(uint32_t b) {
  if (FMT == QMOE_NVFP4) return e4m3_to_f32(b) * 0x1p-120f;  // NaN stays NaN
  return e8m0_to_f32(b);
}

// Largest |x| of `n` bf16 values (bit pattern compare of the magnitudes).
__device__ __forceinline__ uint32_t row_absmax_bits(const uint16_t *src, int n) {
  uint32_t m = 0;
  for (int i = threadIdx.x * 8; i < n; i += kGemvThreads * 8) {
    const uint4 v = *reinterpret_cast<const uint4 *>(src + i);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      m = max(m, w[q] & 0x7FFFu);
      m = max(m, (w[q] >> 16) & 0x7FFFu);
    }
  }
#pragma unroll
  for (int s = 16; s > 0; s >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, s));
  return m;
}

// Power-of-two exponent s with max|x| * 2^-s in [2^14, 2^15) (clamped).
__device__ __forceinline__ int prescale_exponent(uint32_t absmax_bf16_bits) {
  if (absmax_bf16_bits == 0u) return 0;
  const int e = (int)((absmax_bf16_bits >> 7) & 0xFFu) - 127;  // floor(log2) for normal values
  int s = e - 14;
  return max(-100, min(100, s));
}

struct StageShared {
  uint32_t warp_max[kGemvThreads / 32][kRowChunk];
  int shift[kRowChunk];
};

// Stage up to kRowChunk activation rows (bf16, length K) into shared memory as
// fp16 after the per-row power-of-two rescale.  Rows >= nrows are zero.
__device__ void stage_rows(const uint16_t *const *src, int nrows, int K, __half *xs, StageShared &ss) {
  const int w = threadIdx.x >> 5;
  for (int r = 0; r < kRowChunk; ++r) {
    uint32_t m = 0;
    if (r < nrows) m = row_absmax_bits(src[r], K);
    if (lane_id() == 0) ss.warp_max[w][r] = m;
  }
  __syncthreads();
  if (threadIdx.x < kRowChunk) {
    uint32_t m = 0;
    for (int i = 0; i < kGemvThreads / 32; ++i) m = max(m, ss.warp_max[i][threadIdx.x]);
    ss.shift[threadIdx.x] = prescale_exponent(m);
  }
  __syncthreads();
  for (int r = 0; r < kRowChunk; ++r) {
    __half2 *dst = reinterpret_cast<__half2 *>(xs + (size_t)r * K);
    if (r >= nrows) {
      for (int i = threadIdx.x; i < K / 2; i += kGemvThreads) dst[i] = __half2(__float2half(0.f), __float2half(0.f));
      continue;
    }
    const float f = __uint_as_float((uint32_t)(127 - ss.shift[r]) << 23);  // 2^-shift
    for (int i = threadIdx.x * 8; i < K; i += kGemvThreads * 8) {
      const uint4 v = *reinterpret_cast<const uint4 *>(src[r] + i);
      const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float lo = bf16_to_f32(wv[q] & 0xFFFFu) * f, hi = bf16_to_f32(wv[q] >> 16) * f;
        dst[(i >> 1) + q] = __floats2half2_rn(lo, hi);
      }
    }
  }
  __syncthreads();
}

// acc[r][c] (+)= sum over this thread's scale blocks of raw_scale * sum_k x[r][k] * e2m1
template <int FMT, int BS, int RC>
__device__ __forceinline__ void gemv_mainloop(const uint8_t *__restrict__ wexp, const uint8_t *__restrict__ sexp,
                                              int K, int N, int n0, const __half *xs, float (&acc)[RC][8]) {
  const int lane = (int)lane_id();
  const int wi = lane & 7;
  const int kg = ((threadIdx.x >> 5) << 2) | (lane >> 3);
  const int nblocks = K / BS;
  const size_t row_bytes = (size_t)N / 2;
  const uint8_t *wcol = wexp + n0 / 2 + wi * 4;
  const uint8_t *scol = sexp + (size_t)(n0 + wi * 8) * nblocks;
#pragma unroll
  for (int r = 0; r < RC; ++r)
#pragma unroll
    for (int c = 0; c < 8; ++c) acc[r][c] = 0.f;
  for (int b = kg; b < nblocks; b += kKGroups) {
    uint32_t wv[BS];
#pragma unroll
    for (int kk = 0; kk < BS; ++kk)
      wv[kk] = __ldg(reinterpret_cast<const uint32_t *>(wcol + ((size_t)b * BS + kk) * row_bytes));
    uint32_t sb[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) sb[c] = __ldg(scol + (size_t)c * nblocks + b);
    float bp[RC][8];
#pragma unroll
    for (int r = 0; r < RC; ++r)
#pragma unroll
      for (int c = 0; c < 8; ++c) bp[r][c] = 0.f;
    const __half *xb = xs + (size_t)b * BS;
#pragma unroll
    for (int kk = 0; kk < BS; kk += 2) {
      uint32_t x2[RC];
#pragma unroll
      for (int r = 0; r < RC; ++r) x2[r] = *reinterpret_cast<const uint32_t *>(xb + (size_t)r * K + kk);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t wd = wv[kk + h];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint32_t p = e2m1x2_to_f16x2(wd >> (8 * q));
          const uint16_t lo = (uint16_t)(p & 0xFFFFu), hi = (uint16_t)(p >> 16);
#pragma unroll
          for (int r = 0; r < RC; ++r) {
            const uint16_t xv = (uint16_t)(h ? (x2[r] >> 16) : (x2[r] & 0xFFFFu));
            bp[r][2 * q] = fma_f16_f32(lo, xv, bp[r][2 * q]);
            bp[r][2 * q + 1] = fma_f16_f32(hi, xv, bp[r][2 * q + 1]);
          }
        }
      }
    }
    bool special = false;
    float sc[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) sc[c] = raw_scale<FMT>(sb[c], special);
    if (special) {
#pragma unroll
      for (int c = 0; c < 8; ++c) sc[c] = exact_raw_scale<FMT>(sb[c]);
    }
#pragma unroll
    for (int r = 0; r < RC; ++r)
#pragma unroll
      for (int c = 0; c < 8; ++c) acc[r][c] = fmaf(bp[r][c], sc[c], acc[r][c]);
  }
}

// Sum the 32 k-group partials of each (row, column) in a fixed order.
// red: [kKGroups][kRowChunk][kTileN] floats.  Returns via red[0][r][col].
template <int RC>
__device__ __forceinline__ void reduce_kgroups(float (&acc)[RC][8], float *red) {
  const int lane = (int)lane_id();
  const int wi = lane & 7;
  const int kg = ((threadIdx.x >> 5) << 2) | (lane >> 3);
  __syncthreads();  // xs may alias red
#pragma unroll
  for (int r = 0; r < RC; ++r) {
    float4 *d = reinterpret_cast<float4 *>(red + ((size_t)kg * kRowChunk + r) * kTileN + wi * 8);
    d[0] = make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]);
    d[1] = make_float4(acc[r][4], acc[r][5], acc[r][6], acc[r][7]);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < RC * kTileN; i += kGemvThreads) {
    const int r = i / kTileN, col = i % kTileN;
    float s = 0.f;
    for (int g = 0; g < kKGroups; ++g) s += red[((size_t)g * kRowChunk + r) * kTileN + col];
    red[(size_t)r * kTileN + col] = s;
  }
  __syncthreads();
}

__device__ __forceinline__ float swiglu(float gate, float lin, float alpha, float beta, float limit) {
  const float G = fminf(gate, limit);
  const float L = fmaxf(fminf(lin, limit), -limit);
  return G * (1.0f / (1.0f + expf(-alpha * G))) * (L + beta);
}

static size_t gemv_smem_bytes(int K) {
  const size_t xs = (size_t)kRowChunk * K * sizeof(__half);
  const size_t red = (size_t)kKGroups * kRowChunk * kTileN * sizeof(float);
  return xs > red ? xs : red;
}

// FC = 1: K = H, N = 2I, rows read x[token]; output a (bf16, SwiGLU'd).
// FC = 2: K = I, N = H, rows read a[row]; output y (fp32) + un-permute.
template <int FC, int FMT>
__global__ void __launch_bounds__(kGemvThreads, 2) moe_gemv_kernel(GemvArgs g) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  __shared__ StageShared ss;
  __shared__ int is_last;
  constexpr int BS = FMT == QMOE_NVFP4 ? kNvfp4Block : kMxfp4Block;
  const int slot = blockIdx.y;
  const int num_active = g.meta[0];
  if (slot >= num_active) return;
  const int e = g.active[slot];
  const int n0 = blockIdx.x * kTileN;
  const int K = FC == 1 ? g.H : g.I;
  const int N = FC == 1 ? 2 * g.I : g.H;
  const int row0 = g.offsets[e], nrows_all = g.offsets[e + 1] - row0;
  const uint8_t *wexp = (FC == 1 ? g.w1 : g.w2) + (size_t)e * K * (N / 2);
  const uint8_t *sexp = (FC == 1 ? g.s1 : g.s2) + (size_t)e * N * (K / BS);
  const float *gs = FC == 1 ? g.g1 : g.g2;
  const float gscale = gs ? gs[e] : 1.0f;
  __half *xs = reinterpret_cast<__half *>(smem_raw);
  float *red = reinterpret_cast<float *>(smem_raw);

  for (int c0 = 0; c0 < nrows_all; c0 += kRowChunk) {
    const int nrows = min(kRowChunk, nrows_all - c0);
    const uint16_t *src[kRowChunk];
#pragma unroll
    for (int r = 0; r < kRowChunk; ++r) {
      const int p = row0 + c0 + min(r, nrows - 1);
      src[r] = FC == 1 ? g.x + (size_t)(g.p2e[p] / g.k) * g.H : g.a + (size_t)p * g.I;
    }
    stage_rows(src, nrows, K, xs, ss);
    float acc4[4][8];
    if (nrows == 1) {
      float acc[1][8];
      gemv_mainloop<FMT, BS, 1>(wexp, sexp, K, N, n0, xs, acc);
      reduce_kgroups<1>(acc, red);
    } else if (nrows == 2) {
      float acc[2][8];
      gemv_mainloop<FMT, BS, 2>(wexp, sexp, K, N, n0, xs, acc);
      reduce_kgroups<2>(acc, red);
    } else {
      gemv_mainloop<FMT, BS, 4>(wexp, sexp, K, N, n0, xs, acc4);
      reduce_kgroups<4>(acc4, red);
    }
    // epilogue: red[r][col] holds the raw sums of this chunk
    const float fold = FMT == QMOE_NVFP4 ? 0x1p120f : 1.0f;
    if (FC == 1) {
      for (int i = threadIdx.x; i < nrows * (kTileN / 2); i += kGemvThreads) {
        const int r = i / (kTileN / 2), m = i % (kTileN / 2);
        const float un = __uint_as_float((uint32_t)(127 + ss.shift[r]) << 23);
        // fold first: red * 2^120 is the sum in units of the rescaled row, near
        // 2^20 for any row, so undoing the row's 2^-shift afterwards cannot underflow
        const float hg = red[r * kTileN + 2 * m] * fold * un * gscale;
        const float hl = red[r * kTileN + 2 * m + 1] * fold * un * gscale;
        const float act = swiglu(hg, hl, g.alpha, g.beta, g.limit);
        g.a[(size_t)(row0 + c0 + r) * g.I + n0 / 2 + m] = (uint16_t)f32_to_bf16_rne(act);
      }
    } else {
      for (int i = threadIdx.x; i < nrows * kTileN; i += kGemvThreads) {
        const int r = i / kTileN, col = i % kTileN;
        const float un = __uint_as_float((uint32_t)(127 + ss.shift[r]) << 23);
        g.y[(size_t)(row0 + c0 + r) * g.H + n0 + col] = red[r * kTileN + col] * fold * un * gscale;
      }
    }
    __syncthreads();
  }
  if (FC == 2) {
    // last CTA of this column tile forms the weighted un-permute
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) is_last = atomicAdd(&g.counters[blockIdx.x], 1) == num_active - 1;
    __syncthreads();
    if (!is_last) return;
    __threadfence();
    for (int i = threadIdx.x; i < g.T * kTileN; i += kGemvThreads) {
      const int t = i / kTileN, col = i % kTileN;
      float s = 0.f;
      for (int j = 0; j < g.k; ++j) {
        const int ex = t * g.k + j;
        s = fmaf(__ldcg(g.weights + ex), __ldcg(g.y + (size_t)__ldcg(g.e2p + ex) * g.H + n0 + col), s);
      }
      g.out[(size_t)t * g.H + n0 + col] = (uint16_t)f32_to_bf16_rne(s);
    }
  }
}

template <int FC>
static cudaError_t launch_gemv(const GemvArgs &a, cudaStream_t stream) {
  const int K = FC == 1 ? a.H : a.I;
  const int N = FC == 1 ? 2 * a.I : a.H;
  const size_t smem = gemv_smem_bytes(K);
  const int max_slots = a.E < a.T * a.k ? a.E : a.T * a.k;
  dim3 grid(N / kTileN, max_slots);
  // The opt-in shared-memory size is raised only when a larger one is needed,
  // so steady-state calls (and graph capture) make no attribute calls.
  static size_t smem_set[2] = {0, 0};
  const int fi = a.fmt == QMOE_NVFP4 ? 0 : 1;
  auto kfn = a.fmt == QMOE_NVFP4 ? moe_gemv_kernel<FC, QMOE_NVFP4> : moe_gemv_kernel<FC, QMOE_MXFP4>;
  if (smem > 48 * 1024 && smem > smem_set[fi]) {
    cudaError_t err = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    smem_set[fi] = smem;
  }
  kfn<<<grid, kGemvThreads, smem, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_fc1_gemv(const GemvArgs &a, cudaStream_t stream) { return launch_gemv<1>(a, stream); }
cudaError_t launch_fc2_gemv(const GemvArgs &a, cudaStream_t stream) { return launch_gemv<2>(a, stream); }

}  // namespace qmoe
