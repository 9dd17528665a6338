// FP4 (E2M1) -> bf16 weight dequantisation:  packed [E, K, N/2] -> out [E, N, K].
//
// "[CUDA] Coalesce QMoE MXFP4/NVFP4 weight dequantization" (PR #31349) fixes
// what the operation is (nibble selection, block-scale index, output index)
// and the lessons kept here: tile the output so that every packed sector that
// is touched is fully used, emit 16-byte stores so that 8 lanes write one
// 128-byte row segment, read each block scale once per 8 values, and do no
// integer division.  Design here:
//  * a CTA (64 threads) tile is 64 output rows (n) x 64 k; its packed input is
//    64 k rows x 32 bytes, read with 16-byte loads (two per thread) into shared
//    memory whose rows are padded to 9 words and XOR-swizzled so that the
//    transposing reads below are free of bank conflicts;
//  * each thread owns one 32-bit word of codes (8 n) x 8 consecutive k and
//    writes 8 rows x 16 bytes; 8 lanes cover one 128-byte row segment;
//  * CTAs walk the tiles grid-stride (grid = SMs x resident CTAs);
//  * value = round-to-nearest-even bf16 of the exact product e2m1 * scale *
//    global.  With a power-of-two global scale (always for MXFP4 without one)
//    and a normal-range product the fp32 product is exact and its low 16 bits
//    are zero, so the bf16 is just the top half; otherwise the product is
//    formed exactly in fp64 and rounded to bf16 through round-to-odd fp32.
#include <atomic>

#include "qmoe_common.cuh"

namespace qmoe {

constexpr int kDqTileN = 64;
constexpr int kDqTileK = 64;
constexpr int kDqThreads = 64;
constexpr int kDqRowWords = 9;  // 8 data words + 1 pad

// Rows 32..63 of a tile swap word groups 0-3 and 4-7: the 32 reads of a warp
// (8 k chunks x 4 words) then hit 32 distinct banks.
__device__ __forceinline__ int dq_swz(int row) { return ((row >> 5) & 1) << 2; }

// Exact e2m1 code (4 bits) as fp32.  The magnitude bits land where an fp32
// subnormal keeps its top mantissa bits, which is e2m1 * 2^-126 exactly.
__device__ __forceinline__ float e2m1_to_f32(uint32_t code) {
  const uint32_t bits = ((code & 7u) << 22) | ((code & 8u) << 28);
  return __uint_as_float(bits) * 0x1p126f;
}

__device__ __forceinline__ uint32_t exact_product_bf16(float q, float s, float g) {
  // e2m1 (2 significant bits) * scale (<= 4) * global (24): exact in fp64.
  const double d = (double)q * (double)s * (double)g;
  if (d != d) return 0x7FC0u;
  float f = __double2float_rz(d);
  uint32_t u = __float_as_uint(f);
  if ((double)f != d) u |= 1u;  // round to odd keeps the information the bf16 rounding needs
  return (u + 0x7FFFu + ((u >> 16) & 1u)) >> 16;
}

__device__ __forceinline__ bool is_pow2_normal(float g) {
  const uint32_t u = __float_as_uint(g) & 0x7FFFFFFFu;
  return (u & 0x007FFFFFu) == 0u && u >= 0x00800000u && u < 0x7F800000u;
}

template <int FMT>
__global__ void __launch_bounds__(kDqThreads) dequant_kernel(const uint8_t *__restrict__ packed,
                                                            const uint8_t *__restrict__ scales,
                                                            const float *__restrict__ gscale, int E, int N, int K,
                                                            uint16_t *__restrict__ out) {
  constexpr int BS = FMT == QMOE_NVFP4 ? kNvfp4Block : kMxfp4Block;
  __shared__ uint32_t tile[kDqTileK * kDqRowWords];
  const int tid = threadIdx.x;
  const int word = tid >> 3;  // 0..7: n = 8*word + i
  const int c = tid & 7;      // k chunk: k = 8*c + kk
  const int tiles_k = K / kDqTileK, tiles_n = N / kDqTileN;
  const long long ntiles = (long long)E * tiles_n * tiles_k;
  const int nblocks = K / BS;
  const size_t row_bytes = (size_t)N / 2;

  for (long long tileid = blockIdx.x; tileid < ntiles; tileid += gridDim.x) {
    const int tk = (int)(tileid % tiles_k);
    const long long rest = tileid / tiles_k;
    const int tn = (int)(rest % tiles_n);
    const int e = (int)(rest / tiles_n);
    const int k0 = tk * kDqTileK, n0 = tn * kDqTileN;
    // ---- load the packed tile: 64 rows x 32 bytes
    const uint8_t *src = packed + ((size_t)e * K + k0) * row_bytes + n0 / 2;
    uint4 v[2];
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int L = q * kDqThreads + tid, row = L >> 1, half = L & 1;
      v[q] = __ldg(reinterpret_cast<const uint4 *>(src + (size_t)row * row_bytes + half * 16));
    }
    const float gv = gscale ? __ldg(gscale + e) : 1.0f;
    const bool g_fast = gscale == nullptr || is_pow2_normal(gv);
    // block scales of this thread's 8 rows at its k chunk
    uint32_t sb[8];
    const int blk = (k0 + 8 * c) / BS;
#pragma unroll
    for (int i = 0; i < 8; ++i) sb[i] = __ldg(scales + ((size_t)e * N + n0 + 8 * word + i) * nblocks + blk);
    __syncthreads();  // previous tile's reads are done
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int L = q * kDqThreads + tid, row = L >> 1, half = L & 1;
      const uint32_t w4[4] = {v[q].x, v[q].y, v[q].z, v[q].w};
#pragma unroll
      for (int j = 0; j < 4; ++j) tile[row * kDqRowWords + ((half * 4 + j) ^ dq_swz(row))] = w4[j];
    }
    __syncthreads();
    uint32_t wk[8];
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const int row = 8 * c + kk;
      wk[kk] = tile[row * kDqRowWords + (word ^ dq_swz(row))];
    }
    uint16_t *dst = out + ((size_t)e * N + n0 + 8 * word) * K + k0 + 8 * c;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float s = scale_to_f32(FMT, sb[i]);
      const float sg = s * gv;
      const float asg = fabsf(sg);
      const bool fast = g_fast && (sg == 0.0f || (asg >= 0x1p-120f && asg <= 0x1p120f));
      uint32_t o[4];
      if (fast) {
#pragma unroll
        for (int kk = 0; kk < 8; kk += 2) {
          const float p0 = e2m1_to_f32(wk[kk] >> (4 * i)) * sg;
          const float p1 = e2m1_to_f32(wk[kk + 1] >> (4 * i)) * sg;
          o[kk >> 1] = __byte_perm(__float_as_uint(p0), __float_as_uint(p1), 0x7632);
        }
      } else {
#pragma unroll
        for (int kk = 0; kk < 8; kk += 2) {
          const uint32_t b0 = exact_product_bf16(e2m1_to_f32(wk[kk] >> (4 * i)), s, gv);
          const uint32_t b1 = exact_product_bf16(e2m1_to_f32(wk[kk + 1] >> (4 * i)), s, gv);
          o[kk >> 1] = b0 | (b1 << 16);
        }
      }
      *reinterpret_cast<uint4 *>(dst + (size_t)i * K) = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
}

cudaError_t launch_dequant(const uint8_t *packed, const uint8_t *scales, const float *g, int E, int N, int K,
                           int fmt, uint16_t *out, cudaStream_t stream) {
  // resident CTAs per SM, per device and format (0: not yet known)
  static std::atomic<int> blocks_per_sm[kMaxDevices][2];
  const long long ntiles = (long long)E * (N / kDqTileN) * (K / kDqTileK);
  if (ntiles == 0) return cudaSuccess;
  const int dev = current_device();
  if (dev < 0) return cudaErrorInvalidDevice;
  std::atomic<int> &cache = blocks_per_sm[dev][fmt == QMOE_NVFP4 ? 0 : 1];
  int bps = cache.load(std::memory_order_relaxed);
  if (bps == 0) {
    cudaError_t err = fmt == QMOE_NVFP4
                          ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&bps, dequant_kernel<QMOE_NVFP4>, kDqThreads, 0)
                          : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&bps, dequant_kernel<QMOE_MXFP4>, kDqThreads, 0);
    if (err != cudaSuccess) return err;
    if (bps < 1) bps = 1;
    cache.store(bps, std::memory_order_relaxed);
  }
  long long grid = (long long)num_sms() * bps;
  if (grid > ntiles) grid = ntiles;
  if (fmt == QMOE_NVFP4)
    dequant_kernel<QMOE_NVFP4><<<(unsigned)grid, kDqThreads, 0, stream>>>(packed, scales, g, E, N, K, out);
  else
    dequant_kernel<QMOE_MXFP4><<<(unsigned)grid, kDqThreads, 0, stream>>>(packed, scales, g, E, N, K, out);
  return cudaGetLastError();
}

}  // namespace qmoe

namespace qmoe {

// out[e][c][r] = in[e][r][c], bytes unchanged: 64 x 64 byte tiles through
// shared memory (reads along c and writes along r both coalesced), ragged
// edges in both dimensions.  Block scales [E, N, nb] -> [E, nb, N] and back.
constexpr int kTrTile = 64;
constexpr int kTrThreads = 256;

__global__ void __launch_bounds__(kTrThreads) transpose_bytes_kernel(const uint8_t *__restrict__ in, int E, int rows,
                                                                     int cols, uint8_t *__restrict__ out) {
  __shared__ uint8_t t[kTrTile][kTrTile + 4];
  const int tr = (rows + kTrTile - 1) / kTrTile, tc = (cols + kTrTile - 1) / kTrTile;
  const long long ntiles = (long long)E * tr * tc;
  for (long long tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
    const int e = (int)(tile / ((long long)tr * tc));
    const int rem = (int)(tile - (long long)e * tr * tc);
    const int r0 = (rem / tc) * kTrTile, c0 = (rem % tc) * kTrTile;
    const int rh = min(kTrTile, rows - r0), cw = min(kTrTile, cols - c0);
    __syncthreads();  // the previous tile's reads are done
    for (int i = threadIdx.x; i < kTrTile * kTrTile; i += kTrThreads) {
      const int r = i / kTrTile, c = i % kTrTile;
      if (r < rh && c < cw) t[r][c] = in[((size_t)e * rows + r0 + r) * cols + c0 + c];
    }
    __syncthreads();
    for (int i = threadIdx.x; i < kTrTile * kTrTile; i += kTrThreads) {
      const int c = i / kTrTile, r = i % kTrTile;
      if (r < rh && c < cw) out[((size_t)e * cols + c0 + c) * rows + r0 + r] = t[r][c];
    }
  }
}

cudaError_t launch_transpose_bytes(const uint8_t *in, int E, int rows, int cols, uint8_t *out, cudaStream_t stream) {
  const long long ntiles = (long long)E * ((rows + kTrTile - 1) / kTrTile) * ((cols + kTrTile - 1) / kTrTile);
  if (ntiles == 0) return cudaSuccess;
  long long grid = (long long)num_sms() * 8;
  if (grid > ntiles) grid = ntiles;
  transpose_bytes_kernel<<<(unsigned)grid, kTrThreads, 0, stream>>>(in, E, rows, cols, out);
  return cudaGetLastError();
}

}  // namespace qmoe
