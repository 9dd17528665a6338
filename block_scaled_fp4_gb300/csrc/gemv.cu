// Decode GEMVs of the FP4 MoE layer: FC1 (+ SwiGLU) and FC2 (+ weighted
// un-permute), with the E2M1 weights dequantised in registers.
//
// Prior art on the pages ("[CUDA] Speed up the NVFP4 QMoE decode GEMV and
// enable it for MTP verify", PR #31159; operator doc §9b.2/§9b.3): coalesced
// weight and scale streams, weight loads batched ahead of their decode, a
// table-free E2M1 decode, the block scale applied to a per-block partial sum
// instead of to every weight, fp32 accumulation for bf16 activations, and a
// 64-expanded-row window.  Design here (sm_103a):
//  * one CTA = one active expert ("slot") x NT output columns x all of K.
//    256 threads = (NT/8) column words (8 columns = one 32-bit load per k row)
//    x (2048/NT) k-groups; NT in {64, 128, 256} is picked per launch so that
//    the grid holds about two CTAs per SM; a k-group owns whole scale blocks;
//  * two load groups of 16 k rows ping-pong in registers: while one is
//    decoded the next is in flight; the first is issued before the
//    activations are staged;
//  * E2M1 pairs decode with the hardware cvt.rn.f16x2.e2m1x2 (one instruction
//    per two weights) and multiply-accumulate with fma.rn.f32.f16 (fp16
//    operands, exact product, fp32 accumulator);
//  * activations arrive as fp16 rescaled per row by a power of two (largest
//    |x| in [2^14, 2^15)), so every finite bf16 activation is exact in fp16;
//    FC1 takes them from the routing kernel, FC2 rescales its bf16 rows with
//    the row maxima FC1 publishes (atomicMax on fp32 bits: order-free);
//  * the per-block partial sum is multiplied once by the block scale; NVFP4
//    scales are used as E4M3 * 2^-120 (bits moved into fp32 position, exact)
//    and the 2^120 is applied once at the end;
//  * k-group partials are reduced with warp shuffles, then across warps in
//    shared memory, in a fixed order (deterministic).  FC1 applies SwiGLU and
//    writes bf16 activations; FC2 writes fp32 rows and the last CTA to finish
//    a 64-column tile (arrival counter, no waiting) forms
//    out[t] = bf16(sum_j w[t][j] * y[t*k+j]) in fixed j order;
//  * the kernels are chained with programmatic dependent launch: a kernel
//    starts while its predecessor runs and waits (griddepcontrol.wait) before
//    it reads the predecessor's results.
#include <cuda_fp16.h>

#include "qmoe_common.cuh"

namespace qmoe {

constexpr int kGemvThreads = 256;
constexpr int kCounterTile = 64;  // un-permute column tile (counters are per 64 columns)
constexpr int kRowChunk = 2;      // rows decoded together
constexpr int kGroupRows = 16;    // k rows per load group

int gemv_fc2_counter_words(int H) { return H / kCounterTile; }

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

__device__ __forceinline__ float pow2f(int e) { return __uint_as_float((uint32_t)(127 + e) << 23); }

template <int NT>
struct Tile {
  static constexpr int kWords = NT / 8;                   // column words per k row
  static constexpr int kKGroups = kGemvThreads / kWords;  // k-groups in the CTA
  static constexpr int kWarps = kGemvThreads / 32;
};

// Weight rows [k0, k0+16) of this thread's column word, plus (at a block start)
// the block's 8 scale bytes.
struct LoadGroup {
  uint32_t w[kGroupRows];
  uint32_t s[8];
};

template <int BS>
__device__ __forceinline__ void issue_group(LoadGroup &g, const uint8_t *wcol, const uint8_t *scol,
                                            size_t row_bytes, int nblocks, int blk, int sub) {
  const int k0 = blk * BS + sub * kGroupRows;
#pragma unroll
  for (int kk = 0; kk < kGroupRows; ++kk)
    g.w[kk] = __ldg(reinterpret_cast<const uint32_t *>(wcol + (size_t)(k0 + kk) * row_bytes));
  if (sub == 0) {
#pragma unroll
    for (int c = 0; c < 8; ++c) g.s[c] = __ldg(scol + (size_t)c * nblocks + blk);
  }
}

// One load group (16 k rows x 8 columns) decoded and multiplied into the
// block partials bp; at the end of a scale block bp is scaled into acc.
template <int FMT, int RC>
__device__ __forceinline__ void consume_group(const LoadGroup &cur, int sub, const __half *xb, int K,
                                              uint32_t (&sb)[8], float (&bp)[RC][8], float (&acc)[RC][8]) {
  constexpr int BS = FMT == QMOE_NVFP4 ? kNvfp4Block : kMxfp4Block;
  constexpr int G = BS / kGroupRows;
  if (sub == 0) {
    if (G > 1) {  // the scale bytes must outlive this buffer's reuse
#pragma unroll
      for (int c = 0; c < 8; ++c) sb[c] = cur.s[c];
    }
#pragma unroll
    for (int r = 0; r < RC; ++r)
#pragma unroll
      for (int c = 0; c < 8; ++c) bp[r][c] = 0.f;
  }
#pragma unroll
  for (int kk = 0; kk < kGroupRows; kk += 2) {
    uint32_t x2[RC];
#pragma unroll
    for (int r = 0; r < RC; ++r) x2[r] = *reinterpret_cast<const uint32_t *>(xb + (size_t)r * K + kk);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t wd = cur.w[kk + h];
#pragma unroll
      for (int qq = 0; qq < 4; ++qq) {
        const uint32_t p = e2m1x2_to_f16x2(wd >> (8 * qq));
        const uint16_t lo = (uint16_t)(p & 0xFFFFu), hi = (uint16_t)(p >> 16);
#pragma unroll
        for (int r = 0; r < RC; ++r) {
          const uint16_t xv = (uint16_t)(h ? (x2[r] >> 16) : (x2[r] & 0xFFFFu));
          bp[r][2 * qq] = fma_f16_f32(lo, xv, bp[r][2 * qq]);
          bp[r][2 * qq + 1] = fma_f16_f32(hi, xv, bp[r][2 * qq + 1]);
        }
      }
    }
  }
  if (sub == G - 1) {
    bool special = false;
    float sc[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) sc[c] = raw_scale<FMT>(G > 1 ? sb[c] : cur.s[c], special);
    if (special) {
#pragma unroll
      for (int c = 0; c < 8; ++c) sc[c] = exact_raw_scale<FMT>(G > 1 ? sb[c] : cur.s[c]);
    }
#pragma unroll
    for (int r = 0; r < RC; ++r)
#pragma unroll
      for (int c = 0; c < 8; ++c) acc[r][c] = fmaf(bp[r][c], sc[c], acc[r][c]);
  }
}

// acc[r][c] = sum over this thread's scale blocks of raw_scale * sum_k x[r][k] * e2m1.
// Two load groups ping-pong: while one is decoded the other is in flight.
// `ga` already holds the first group.
template <int FMT, int NT, int RC>
__device__ __forceinline__ void gemv_mainloop(const uint8_t *__restrict__ wexp, const uint8_t *__restrict__ sexp,
                                              int K, int N, int n0, const __half *xs, LoadGroup &ga,
                                              float (&acc)[RC][8]) {
  constexpr int BS = FMT == QMOE_NVFP4 ? kNvfp4Block : kMxfp4Block;
  constexpr int G = BS / kGroupRows;  // load groups per scale block
  using T = Tile<NT>;
  const int wi = threadIdx.x % T::kWords;
  const int kg = threadIdx.x / T::kWords;
  const int nblocks = K / BS;
  const size_t row_bytes = (size_t)N / 2;
  const uint8_t *wcol = wexp + n0 / 2 + wi * 4;
  const uint8_t *scol = sexp + (size_t)(n0 + wi * 8) * nblocks;
  const int my_blocks = kg < nblocks ? (nblocks - 1 - kg) / T::kKGroups + 1 : 0;
  const int nq = my_blocks * G;
#pragma unroll
  for (int r = 0; r < RC; ++r)
#pragma unroll
    for (int c = 0; c < 8; ++c) acc[r][c] = 0.f;
  LoadGroup gb;
  uint32_t sb[8];
  float bp[RC][8];
  for (int q = 0; q < nq; q += 2) {
    if (q + 1 < nq)
      issue_group<BS>(gb, wcol, scol, row_bytes, nblocks, kg + ((q + 1) / G) * T::kKGroups, (q + 1) % G);
    consume_group<FMT, RC>(ga, q % G, xs + (size_t)(kg + (q / G) * T::kKGroups) * BS + (q % G) * kGroupRows, K,
                           sb, bp, acc);
    if (q + 1 >= nq) break;
    if (q + 2 < nq)
      issue_group<BS>(ga, wcol, scol, row_bytes, nblocks, kg + ((q + 2) / G) * T::kKGroups, (q + 2) % G);
    consume_group<FMT, RC>(gb, (q + 1) % G,
                           xs + (size_t)(kg + ((q + 1) / G) * T::kKGroups) * BS + ((q + 1) % G) * kGroupRows, K,
                           sb, bp, acc);
  }
}

// Sum the k-group partials of each (row, column) in a fixed order: shuffles
// inside a warp, then the warps' partials in shared memory (red: [warps][rows][NT]).
// The result is left in red[r * NT + col].
template <int NT, int RC>
__device__ __forceinline__ void reduce_kgroups(float (&acc)[RC][8], float *red) {
  using T = Tile<NT>;
  constexpr int kPer = (RC * NT + kGemvThreads - 1) / kGemvThreads;
  const int lane = (int)lane_id(), warp = threadIdx.x >> 5;
#pragma unroll
  for (int m = T::kWords; m < 32; m <<= 1)
#pragma unroll
    for (int r = 0; r < RC; ++r)
#pragma unroll
      for (int c = 0; c < 8; ++c) acc[r][c] += __shfl_xor_sync(0xFFFFFFFFu, acc[r][c], m);
  __syncthreads();  // the staged activations (aliasing red) are no longer read
  if (lane < T::kWords) {
#pragma unroll
    for (int r = 0; r < RC; ++r) {
      float4 *d = reinterpret_cast<float4 *>(red + ((size_t)warp * kRowChunk + r) * NT + lane * 8);
      d[0] = make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]);
      d[1] = make_float4(acc[r][4], acc[r][5], acc[r][6], acc[r][7]);
    }
  }
  __syncthreads();
  float s[kPer];
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int i = threadIdx.x + j * kGemvThreads;
    s[j] = 0.f;
    if (i < RC * NT) {
      const int r = i / NT, col = i % NT;
      for (int w = 0; w < T::kWarps; ++w) s[j] += red[((size_t)w * kRowChunk + r) * NT + col];
    }
  }
  __syncthreads();
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int i = threadIdx.x + j * kGemvThreads;
    if (i < RC * NT) red[i] = s[j];
  }
  __syncthreads();
}

__device__ __forceinline__ float swiglu(float gate, float lin, float alpha, float beta, float limit) {
  const float G = fminf(gate, limit);
  const float L = fmaxf(fminf(lin, limit), -limit);
  return G * (1.0f / (1.0f + expf(-alpha * G))) * (L + beta);
}

template <int NT>
static size_t gemv_smem_bytes(int K) {
  const size_t xs = (size_t)kRowChunk * K * sizeof(__half);
  const size_t red = (size_t)Tile<NT>::kWarps * kRowChunk * NT * sizeof(float);
  return xs > red ? xs : red;
}

// Stage activation rows [c0, c0 + nrows) of the slot into shared memory (fp16,
// rescaled).  FC1: copies of the token rows the routing kernel converted.
// FC2: the bf16 rows of a, rescaled with the row maxima FC1 published.
// shifts[r] receive the exponents to undo.
template <int FC>
__device__ __forceinline__ void stage_rows(const GemvArgs &g, const SlotDesc &sd, int c0, int nrows, int K,
                                           __half *xs, int *shifts) {
  if (threadIdx.x < kRowChunk) {
    int sh = 0;
    if ((int)threadIdx.x < nrows) {
      const int p = sd.row0 + c0 + threadIdx.x;
      if (FC == 1) {
        sh = g.xshift[g.p2e[p] / g.k];
      } else {
        const uint32_t m = __ldcg(g.rowmax + p);
        if (m != 0u) sh = max(-100, min(100, (int)((m >> 23) & 0xFFu) - 127 - 14));
      }
    }
    shifts[threadIdx.x] = sh;
  }
  __syncthreads();
  for (int r = 0; r < kRowChunk; ++r) {
    uint4 *dst = reinterpret_cast<uint4 *>(xs + (size_t)r * K);
    if (r >= nrows) {
      for (int i = threadIdx.x; i < K / 8; i += kGemvThreads) dst[i] = make_uint4(0, 0, 0, 0);
      continue;
    }
    const int p = sd.row0 + c0 + r;
    if (FC == 1) {
      const uint4 *src = reinterpret_cast<const uint4 *>(g.x16 + (size_t)(g.p2e[p] / g.k) * g.H);
      for (int i = threadIdx.x; i < K / 8; i += kGemvThreads) dst[i] = __ldcg(src + i);
    } else {
      const uint4 *src = reinterpret_cast<const uint4 *>(g.a + (size_t)p * g.I);
      const float f = pow2f(-shifts[r]);
      for (int i = threadIdx.x; i < K / 8; i += kGemvThreads) {
        const uint4 v = __ldcg(src + i);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t o[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const __half2 h = __floats2half2_rn(bf16_to_f32(w[q] & 0xFFFFu) * f, bf16_to_f32(w[q] >> 16) * f);
          o[q] = *reinterpret_cast<const uint32_t *>(&h);
        }
        dst[i] = make_uint4(o[0], o[1], o[2], o[3]);
      }
    }
  }
  __syncthreads();
}

// FC = 1: K = H, N = 2I, rows read x16[token]; output a (bf16, SwiGLU'd).
// FC = 2: K = I, N = H, rows read a[row]; output y (fp32) + un-permute.
template <int FC, int FMT, int NT>
__global__ void __launch_bounds__(kGemvThreads, 2) moe_gemv_kernel(GemvArgs g) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  __shared__ int shifts[kRowChunk];
  __shared__ int is_last;
  constexpr int BS = FMT == QMOE_NVFP4 ? kNvfp4Block : kMxfp4Block;
  using T = Tile<NT>;
  pdl_wait();  // routing (and for FC2 also FC1) results are visible from here on
  if (FC == 1) pdl_launch_dependents();
  const int slot = blockIdx.y;
  if (slot >= g.meta[0]) return;
  const SlotDesc sd = g.slots[slot];
  const int e = sd.e;
  const int n0 = blockIdx.x * NT;
  const int K = FC == 1 ? g.H : g.I;
  const int N = FC == 1 ? 2 * g.I : g.H;
  const uint8_t *wexp = (FC == 1 ? g.w1 : g.w2) + (size_t)e * K * (N / 2);
  const uint8_t *sexp = (FC == 1 ? g.s1 : g.s2) + (size_t)e * N * (K / BS);
  const float *gs = FC == 1 ? g.g1 : g.g2;
  const float gscale = gs ? gs[e] : 1.0f;
  __half *xs = reinterpret_cast<__half *>(smem_raw);
  float *red = reinterpret_cast<float *>(smem_raw);
  const int wi = threadIdx.x % T::kWords, kg = threadIdx.x / T::kWords;
  const int nblocks = K / BS;

  for (int c0 = 0; c0 < sd.nrows; c0 += kRowChunk) {
    const int nrows = min(kRowChunk, sd.nrows - c0);
    // first weight group in flight before the activations are staged
    LoadGroup first;
    if (kg < nblocks)
      issue_group<BS>(first, wexp + n0 / 2 + wi * 4, sexp + (size_t)(n0 + wi * 8) * nblocks, (size_t)N / 2,
                      nblocks, kg, 0);
    stage_rows<FC>(g, sd, c0, nrows, K, xs, shifts);
    if (nrows == 1) {
      float acc[1][8];
      gemv_mainloop<FMT, NT, 1>(wexp, sexp, K, N, n0, xs, first, acc);
      reduce_kgroups<NT, 1>(acc, red);
    } else {
      float acc[2][8];
      gemv_mainloop<FMT, NT, 2>(wexp, sexp, K, N, n0, xs, first, acc);
      reduce_kgroups<NT, 2>(acc, red);
    }
    // epilogue: red[r * NT + col] holds the raw sums of this chunk.  The 2^120
    // fold comes first so that undoing the row's 2^-shift cannot underflow.
    const float fold = FMT == QMOE_NVFP4 ? 0x1p120f : 1.0f;
    if (FC == 1) {
      for (int i = threadIdx.x; i < nrows * (NT / 2); i += kGemvThreads) {
        const int r = i / (NT / 2), m = i % (NT / 2);
        const float un = pow2f(shifts[r]);
        const float hg = red[r * NT + 2 * m] * fold * un * gscale;
        const float hl = red[r * NT + 2 * m + 1] * fold * un * gscale;
        const uint32_t ab = f32_to_bf16_rne(swiglu(hg, hl, g.alpha, g.beta, g.limit));
        const int p = sd.row0 + c0 + r;
        g.a[(size_t)p * g.I + n0 / 2 + m] = (uint16_t)ab;
        // NT / 2 >= 32 and nrows * NT / 2 is a multiple of 32: a warp is either
        // wholly inside this loop iteration and shares one row r, or outside it
        const uint32_t mag = __reduce_max_sync(0xFFFFFFFFu, (ab & 0x7FFFu) << 16);
        if (lane_id() == 0) atomicMax(g.rowmax + p, mag);
      }
    } else {
      for (int i = threadIdx.x; i < nrows * NT; i += kGemvThreads) {
        const int r = i / NT, col = i % NT;
        const float un = pow2f(shifts[r]);
        g.y[(size_t)(sd.row0 + c0 + r) * g.H + n0 + col] = red[r * NT + col] * fold * un * gscale;
      }
    }
    __syncthreads();
  }
  if (FC == 2) {
    // the last CTA of each 64-column un-permute tile forms the weighted sum
    __threadfence();
    __syncthreads();
    for (int t0 = 0; t0 < NT; t0 += kCounterTile) {
      const int tile = (n0 + t0) / kCounterTile;
      if (threadIdx.x == 0) is_last = atomicAdd(&g.counters[tile], 1) == g.meta[0] - 1;
      __syncthreads();
      if (is_last) {
        __threadfence();
        for (int i = threadIdx.x; i < g.T * kCounterTile; i += kGemvThreads) {
          const int t = i / kCounterTile, col = n0 + t0 + i % kCounterTile;
          float s = 0.f;
          for (int j = 0; j < g.k; ++j) {
            const int ex = t * g.k + j;
            s = fmaf(__ldcg(g.weights + ex), __ldcg(g.y + (size_t)__ldcg(g.e2p + ex) * g.H + col), s);
          }
          g.out[(size_t)t * g.H + col] = (uint16_t)f32_to_bf16_rne(s);
        }
      }
      __syncthreads();
    }
  }
}

template <int FC, int FMT, int NT>
static cudaError_t launch_one(const GemvArgs &a, dim3 grid, size_t smem, cudaStream_t stream) {
  // The opt-in shared-memory size is raised only when a larger one is needed,
  // so steady-state calls (and graph capture) make no attribute calls.
  static size_t smem_set = 0;
  auto kfn = moe_gemv_kernel<FC, FMT, NT>;
  if (smem > 48 * 1024 && smem > smem_set) {
    cudaError_t err = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    smem_set = smem;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kGemvThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kfn, a);
}

// Widest column tile that still gives about two CTAs per SM.
static int pick_tile(int N, int slots) {
  const int target = 2 * num_sms();
  for (int nt : {256, 128}) {
    if (N % nt == 0 && (long long)slots * (N / nt) >= target) return nt;
  }
  return 64;
}

template <int FC>
static cudaError_t launch_gemv(const GemvArgs &a, cudaStream_t stream) {
  const int K = FC == 1 ? a.H : a.I;
  const int N = FC == 1 ? 2 * a.I : a.H;
  const int slots = a.E < a.T * a.k ? a.E : a.T * a.k;
  const int nt = pick_tile(N, slots);
  const dim3 grid(N / nt, slots);
  if (a.fmt == QMOE_NVFP4) {
    if (nt == 256) return launch_one<FC, QMOE_NVFP4, 256>(a, grid, gemv_smem_bytes<256>(K), stream);
    if (nt == 128) return launch_one<FC, QMOE_NVFP4, 128>(a, grid, gemv_smem_bytes<128>(K), stream);
    return launch_one<FC, QMOE_NVFP4, 64>(a, grid, gemv_smem_bytes<64>(K), stream);
  }
  if (nt == 256) return launch_one<FC, QMOE_MXFP4, 256>(a, grid, gemv_smem_bytes<256>(K), stream);
  if (nt == 128) return launch_one<FC, QMOE_MXFP4, 128>(a, grid, gemv_smem_bytes<128>(K), stream);
  return launch_one<FC, QMOE_MXFP4, 64>(a, grid, gemv_smem_bytes<64>(K), stream);
}

cudaError_t launch_fc1_gemv(const GemvArgs &a, cudaStream_t stream) { return launch_gemv<1>(a, stream); }
cudaError_t launch_fc2_gemv(const GemvArgs &a, cudaStream_t stream) { return launch_gemv<2>(a, stream); }

}  // namespace qmoe
