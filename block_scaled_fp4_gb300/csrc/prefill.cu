// Prefill path of the FP4 MoE layer (more than 64 expanded rows): the expert
// weights are dequantised to bf16 ("[CUDA] Coalesce QMoE MXFP4/NVFP4 weight
// dequantization", PR #31349; "MoE and QMoE - CUDA Operator Documentation"
// §4.3, §9b.1), then two grouped GEMMs run on the tensor cores and a last
// kernel forms the weighted sum over each token's experts (§1 pipeline:
// GEMM1 -> activation -> GEMM2 -> un-permute -> weighted sum).
//
// Grouped GEMM (bf16 operands, fp32 accumulation, mma.sync m16n8k16):
//  * the rows of every expert are contiguous in expert order (the permute
//    maps); a CTA computes a 128-row x 128-column tile of one expert, the
//    tiles of all experts numbered expert by expert (each CTA finds its own
//    from the expert offsets with a warp prefix sum);
//  * GEMM1's left operand is gathered on the fly: permuted row p reads token
//    perm_to_expanded[p] / k of x (no expanded copy of the activations);
//  * operands are staged by cp.async (16 bytes per thread, zero-filled past
//    the expert's last row) into a 3-stage ring of 128 x 32 bf16 tiles whose
//    16-byte chunks are XOR-swizzled so that ldmatrix reads are free of bank
//    conflicts;
//  * 8 warps, each a 32 x 64 sub-tile (2 x 8 m16n8 accumulators);
//  * GEMM1's epilogue applies SwiGLU to the adjacent (gate, linear) columns
//    that an accumulator fragment holds and writes a = bf16(SwiGLU) [R, I];
//    GEMM2's writes y (fp32) [R, H].
#include "qmoe_common.cuh"

namespace qmoe {

constexpr int kBM = 128, kBN = 128, kBK = 32, kStages = 3, kGemmThreads = 256;
constexpr int kTileA = kBM * kBK;  // bf16 elements of one stage's left tile
constexpr int kTileB = kBN * kBK;
constexpr int kGemmSmem = kStages * (kTileA + kTileB) * 2;

struct GroupedGemm {
  const uint16_t *A;       // bf16 left-operand rows
  const int32_t *perm;     // non-null: row p of the expert order reads A row perm[p] / ktop
  int ktop;
  int lda;                 // elements between rows of A
  const uint16_t *B;       // bf16 [E, N, K]: row n of expert e holds its K weights
  const int32_t *offsets;  // [E + 1] first row of each expert
  int E, N, K;
  int swiglu;              // 1: out_a[p][n / 2] = bf16(SwiGLU(h[n], h[n + 1])); 0: out_y[p][n] = h
  uint16_t *out_a;         // [R, N / 2]
  float *out_y;            // [R, N]
  float alpha, beta, limit;
};

__device__ __forceinline__ uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

// 16-byte async copy; src_bytes = 0 fills the destination with zeros.
__device__ __forceinline__ void cp_async16_zfill(uint32_t dst, const void *src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// Element offset of 16-byte chunk c of row r in a swizzled [rows][kBK] tile.
__device__ __forceinline__ int swz(int r, int c) { return r * kBK + ((c ^ ((r >> 1) & 3)) << 3); }

__global__ void __launch_bounds__(kGemmThreads) grouped_gemm_kernel(const __grid_constant__ GroupedGemm p) {
  extern __shared__ __align__(128) uint16_t gsm[];
  __shared__ int s_e, s_row0, s_rows;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // this CTA's (expert, row tile): tiles of expert e are [pre_e, pre_e + ceil(rows_e / kBM))
  if (warp == 0) {
    const int per = (p.E + 31) / 32;
    int sum = 0;
    for (int q = 0; q < per; ++q) {
      const int e = lane * per + q;
      if (e < p.E) sum += (__ldg(p.offsets + e + 1) - __ldg(p.offsets + e) + kBM - 1) / kBM;
    }
    int incl = sum;
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
      const int v = __shfl_up_sync(0xFFFFFFFFu, incl, m);
      if (lane >= m) incl += v;
    }
    const int total = __shfl_sync(0xFFFFFFFFu, incl, 31);
    const int bx = (int)blockIdx.x;
    int run = incl - sum;
    for (int q = 0; q < per; ++q) {
      const int e = lane * per + q;
      if (e < p.E) {
        const int o0 = __ldg(p.offsets + e), o1 = __ldg(p.offsets + e + 1);
        const int c = (o1 - o0 + kBM - 1) / kBM;
        if (bx >= run && bx < run + c) {
          s_e = e;
          s_row0 = o0 + (bx - run) * kBM;
          s_rows = min(kBM, o1 - s_row0);
        }
        run += c;
      }
    }
    __syncwarp();
    if (lane == 0 && bx >= total) s_e = -1;  // more CTAs than tiles
  }
  __syncthreads();
  const int e = s_e;
  if (e < 0) return;
  const int row0 = s_row0, rows = s_rows;
  const int n0 = (int)blockIdx.y * kBN;
  const int KT = p.K / kBK;

  auto load_stage = [&](int st, int k0) {
    uint16_t *As = gsm + st * (kTileA + kTileB);
    uint16_t *Bs = As + kTileA;
    for (int i = tid; i < kBM * 4; i += kGemmThreads) {
      const int r = i >> 2, c = i & 3;
      const uint16_t *src = p.A;
      uint32_t bytes = 0;
      if (r < rows) {
        const int g = row0 + r;
        const int arow = p.perm ? __ldg(p.perm + g) / p.ktop : g;
        src = p.A + (size_t)arow * p.lda + k0 + c * 8;
        bytes = 16;
      }
      cp_async16_zfill(smem_u32(As + swz(r, c)), src, bytes);
    }
    for (int i = tid; i < kBN * 4; i += kGemmThreads) {
      const int r = i >> 2, c = i & 3;
      const uint16_t *src = p.B;
      uint32_t bytes = 0;
      if (n0 + r < p.N) {
        src = p.B + ((size_t)e * p.N + n0 + r) * p.K + k0 + c * 8;
        bytes = 16;
      }
      cp_async16_zfill(smem_u32(Bs + swz(r, c)), src, bytes);
    }
  };

  float acc[2][8][4];
#pragma unroll
  for (int mi = 0; mi < 2; ++mi)
#pragma unroll
    for (int ni = 0; ni < 8; ++ni)
#pragma unroll
      for (int q = 0; q < 4; ++q) acc[mi][ni][q] = 0.f;

#pragma unroll
  for (int s = 0; s < kStages - 1; ++s) {
    if (s < KT) load_stage(s, s * kBK);
    cp_async_commit();
  }
  const int wm = warp & 3, wn = warp >> 2;  // 4 x 2 warps of 32 x 64
  for (int kt = 0; kt < KT; ++kt) {
    cp_async_wait<kStages - 2>();
    __syncthreads();  // stage kt landed for every thread; stage kt - 1 is no longer read
    {
      const int nk = kt + kStages - 1;
      if (nk < KT) load_stage(nk % kStages, nk * kBK);
      cp_async_commit();
    }
    const uint16_t *As = gsm + (kt % kStages) * (kTileA + kTileB);
    const uint16_t *Bs = As + kTileA;
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
      uint32_t a[2][4], b[8][2];
#pragma unroll
      for (int mi = 0; mi < 2; ++mi) {
        const int r = wm * 32 + mi * 16 + (lane & 15);
        ldmatrix_x4(smem_u32(As + swz(r, ks * 2 + (lane >> 4))), a[mi]);
      }
#pragma unroll
      for (int nj = 0; nj < 4; ++nj) {
        const int r = wn * 64 + nj * 16 + (lane & 7) + ((lane >> 4) << 3);
        uint32_t t4[4];
        ldmatrix_x4(smem_u32(Bs + swz(r, ks * 2 + ((lane >> 3) & 1))), t4);
        b[2 * nj][0] = t4[0];
        b[2 * nj][1] = t4[1];
        b[2 * nj + 1][0] = t4[2];
        b[2 * nj + 1][1] = t4[3];
      }
#pragma unroll
      for (int mi = 0; mi < 2; ++mi)
#pragma unroll
        for (int ni = 0; ni < 8; ++ni) mma_bf16(acc[mi][ni], a[mi], b[ni][0], b[ni][1]);
    }
  }
  cp_async_wait<0>();

  // epilogue: fragment (mi, ni) holds rows r, r + 8 and the column pair (c, c + 1)
#pragma unroll
  for (int mi = 0; mi < 2; ++mi) {
#pragma unroll
    for (int ni = 0; ni < 8; ++ni) {
      const int c = n0 + wn * 64 + ni * 8 + 2 * (lane & 3);
      if (c >= p.N) continue;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int r = wm * 32 + mi * 16 + (lane >> 2) + 8 * h;
        if (r >= rows) continue;
        const float v0 = acc[mi][ni][2 * h], v1 = acc[mi][ni][2 * h + 1];
        const size_t prow = (size_t)(row0 + r);
        if (p.swiglu) {
          p.out_a[prow * (p.N / 2) + c / 2] = (uint16_t)f32_to_bf16_rne(swiglu(v0, v1, p.alpha, p.beta, p.limit));
        } else {
          *reinterpret_cast<float2 *>(p.out_y + prow * p.N + c) = make_float2(v0, v1);
        }
      }
    }
  }
}

// out[t][h] = bf16(sum_j w[t][j] * y[expanded_to_perm[t * k + j]][h]), j in order.
__global__ void __launch_bounds__(256) unpermute_kernel(const float *__restrict__ y, const int32_t *__restrict__ e2p,
                                                        const float *__restrict__ w, int T, int H, int k,
                                                        uint16_t *__restrict__ out) {
  const int half = H / 2;
  const long long n = (long long)T * half;
  for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < n;
       idx += (long long)gridDim.x * blockDim.x) {
    const int t = (int)(idx / half), h = 2 * (int)(idx - (long long)t * half);
    float s0 = 0.f, s1 = 0.f;
    for (int j = 0; j < k; ++j) {
      const int pr = __ldg(e2p + t * k + j);
      const float2 v = *reinterpret_cast<const float2 *>(y + (size_t)pr * H + h);
      const float wt = __ldg(w + t * k + j);
      s0 = fmaf(wt, v.x, s0);
      s1 = fmaf(wt, v.y, s1);
    }
    reinterpret_cast<uint32_t *>(out + (size_t)t * H)[h / 2] = f32_to_bf16_rne(s0) | (f32_to_bf16_rne(s1) << 16);
  }
}

cudaError_t launch_prefill(const PrefillArgs &a, cudaStream_t stream) {
  static bool smem_set = false;
  if (!smem_set) {
    cudaError_t err = cudaFuncSetAttribute(grouped_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kGemmSmem);
    if (err != cudaSuccess) return err;
    smem_set = true;
  }
  const int R = a.T * a.k;
  const int na_max = a.E < R ? a.E : R;
  const unsigned mtiles = (unsigned)((R + kBM - 1) / kBM + na_max);  // >= the sum over experts of ceil(rows / kBM)
  GroupedGemm g1{};
  g1.A = a.x; g1.perm = a.p2e; g1.ktop = a.k; g1.lda = a.H;
  g1.B = a.w1d; g1.offsets = a.offsets; g1.E = a.E; g1.N = 2 * a.I; g1.K = a.H;
  g1.swiglu = 1; g1.out_a = a.act; g1.alpha = a.alpha; g1.beta = a.beta; g1.limit = a.limit;
  grouped_gemm_kernel<<<dim3(mtiles, (unsigned)((g1.N + kBN - 1) / kBN)), kGemmThreads, kGemmSmem, stream>>>(g1);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  GroupedGemm g2{};
  g2.A = a.act; g2.perm = nullptr; g2.ktop = 1; g2.lda = a.I;
  g2.B = a.w2d; g2.offsets = a.offsets; g2.E = a.E; g2.N = a.H; g2.K = a.I;
  g2.swiglu = 0; g2.out_y = a.y;
  grouped_gemm_kernel<<<dim3(mtiles, (unsigned)((g2.N + kBN - 1) / kBN)), kGemmThreads, kGemmSmem, stream>>>(g2);
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  const long long work = (long long)a.T * (a.H / 2);
  long long grid = (work + 255) / 256;
  if (grid > (long long)num_sms() * 8) grid = (long long)num_sms() * 8;
  unpermute_kernel<<<(unsigned)grid, 256, 0, stream>>>(a.y, a.e2p, a.weights, a.T, a.H, a.k, a.out);
  return cudaGetLastError();
}

}  // namespace qmoe
