// Prefill path of the FP4 MoE layer (more than 64 expanded rows), after the
// routing ("MoE and QMoE - CUDA Operator Documentation" §1 pipeline: GEMM1 ->
// activation -> GEMM2 -> un-permute -> weighted sum):
//  * gather_rows_kernel puts the token rows in expert order for FC1;
//  * per FC, the fused W4A16 grouped GEMM of prefill_fp4.cu over the packed
//    weights, or -- when the caller gives bf16 weights dequantised by
//    qmoe_fp4_dequant ("[CUDA] Coalesce QMoE MXFP4/NVFP4 weight
//    dequantization", PR #31349; §4.3, §9b.1) -- grouped_gemm_tc_kernel below;
//  * unpermute_kernel forms the weighted sum over each token's experts.
//
// grouped_gemm_tc_kernel: bf16 operands, fp32 accumulation on the
// 5th-generation tensor cores (tcgen05.mma, accumulator in tensor memory);
// the rows of every expert are contiguous in expert order (the permute maps)
// and a CTA computes a 128-row x 128-column tile of one expert, the tiles of
// all experts numbered expert by expert.  GEMM1's left operand is gathered
// on the fly (permuted row p reads token perm_to_expanded[p] / k of x) and
// its epilogue applies SwiGLU to the (gate, linear) columns of a row,
// writing a = bf16(SwiGLU) [R, I]; GEMM2 writes y (fp32) [R, H].
#include <atomic>

#include "qmoe_common.cuh"

namespace qmoe {

struct GroupedGemm {
  const uint16_t *A;       // bf16 left-operand rows
  const int32_t *perm;     // non-null: row p of the expert order reads A row perm[p] / ktop
  int ktop;
  int lda;                 // elements between rows of A
  const uint16_t *B;       // bf16 [E, N, K]: row n of expert e holds its K weights
  const int32_t *offsets;  // [E + 1] first row of each expert
  int E, N, K;
  int swiglu;              // 1: out_a[p][n / 2] = bf16(SwiGLU(h[n], h[n + 1])); 0: out_y[p][n] = h
  int concat;              // with swiglu: B holds the gate rows [0, N/2) then the linear rows [N/2, N);
                           // output column n reads row n / 2 (n even) or N / 2 + n / 2 (n odd)
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
// ---- tcgen05 grouped GEMM ------------------------------------------------------
//
// The same grouped GEMM on the 5th-generation tensor cores: a CTA of 4 warps
// computes a 128 x 128 tile with tcgen05.mma (kind::f16, bf16 operands, fp32
// accumulator in tensor memory, M = 128, N = 128, K = 16 per instruction).
//  * operands: 3-stage ring of 128 x 64 bf16 tiles per operand, K-major with
//    the 128-byte swizzle (16-byte chunk c of row r at r * 128 + ((c ^ (r & 7))
//    * 16), 8-row groups 1 KB apart); filled by cp.async from every thread (the
//    left operand's rows gathered), made visible to the tensor core with
//    fence.proxy.async before the barrier that precedes the MMA issue;
//  * one thread issues the 4 MMAs of a stage and tcgen05.commit's an mbarrier,
//    which releases the stage for its next fill;
//  * epilogue: each warp reads its 32 accumulator rows (tensor-memory lanes
//    32w..32w+31) 32 columns at a time with tcgen05.ld, applies SwiGLU (first
//    GEMM) and stores;
//  * every wait is bounded; the tensor memory is always released.
constexpr int kTcBM = 128, kTcBN = 128, kTcBK = 64, kTcStages = 3, kTcThreads = 128;
constexpr int kTcTileBytes = kTcBM * kTcBK * 2;                      // 16 KB per operand tile
constexpr int kTcSmem = kTcStages * 2 * kTcTileBytes + 1024;         // + room to align to 1 KB
constexpr uint32_t kTcWaitLimit = 1u << 22;
// instruction descriptor: fp32 accumulator (bits 4-5 = 1), bf16 A (bits 7-9 = 1)
// and B (bits 10-12 = 1), both K-major, N >> 3 at bit 17, M >> 4 at bit 24
constexpr uint32_t kTcIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kTcBN >> 3) << 17) |
                              ((uint32_t)(kTcBM >> 4) << 24);
static_assert(kTcBM == 128 && kTcBN % 16 == 0 && kTcBN <= 256, "tcgen05.mma M = 128 shape");

// Shared-memory matrix descriptor of a K-major, 128-byte-swizzled tile: start
// address >> 4 (bits 0-13), leading byte offset 16 (unused with this swizzle),
// stride byte offset 1024 between 8-row groups (bits 32-45), descriptor
// version 1 (bits 46-47), swizzle mode 128 B (value 2, bits 61-63).
__device__ __forceinline__ uint64_t tc_desc_sw128(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
__device__ __forceinline__ uint32_t tc_sw128(int r, int c) { return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4)); }

__device__ __forceinline__ void tc_mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ bool tc_mbar_wait(uint64_t *bar, uint32_t parity) {
  for (uint32_t i = 0; i < kTcWaitLimit; ++i) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    if (done) return true;
  }
  return false;
}

__global__ void __launch_bounds__(kTcThreads) grouped_gemm_tc_kernel(const __grid_constant__ GroupedGemm p,
                                                                    int32_t *err_flag) {
  extern __shared__ __align__(1024) unsigned char tsm[];
  __shared__ uint64_t mma_done[kTcStages];
  __shared__ uint32_t tmem_base_s;
  __shared__ int s_e, s_row0, s_rows, s_abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (warp == 0) {  // this CTA's (expert, row tile), as in the mma.sync kernel
    const int per = (p.E + 31) / 32;
    int sum = 0;
    for (int q = 0; q < per; ++q) {
      const int e = lane * per + q;
      if (e < p.E) sum += (__ldg(p.offsets + e + 1) - __ldg(p.offsets + e) + kTcBM - 1) / kTcBM;
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
        const int c = (o1 - o0 + kTcBM - 1) / kTcBM;
        if (bx >= run && bx < run + c) {
          s_e = e;
          s_row0 = o0 + (bx - run) * kTcBM;
          s_rows = min(kTcBM, o1 - s_row0);
        }
        run += c;
      }
    }
    __syncwarp();
    if (lane == 0) {
      if (bx >= total) s_e = -1;
      s_abort = 0;
    }
  }
  __syncthreads();
  const int e = s_e;
  if (e < 0) return;  // CTA-uniform, before any tensor memory is held
  const int row0 = s_row0, rows = s_rows;
  const int n0 = (int)blockIdx.y * kTcBN;
  const int KT = p.K / kTcBK;
  unsigned char *base = tsm + ((1024u - (smem_u32(tsm) & 1023u)) & 1023u);

  if (warp == 0) {  // 128 fp32 columns of tensor memory: the 128 x 128 accumulator
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_base_s)),
                 "r"(128u)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (tid == 32) {
    for (int i = 0; i < kTcStages; ++i) tc_mbar_init(&mma_done[i], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = tmem_base_s;

  // The rows a thread copies are the same at every k step (row (tid >> 3) +
  // 16 q, chunk tid & 7): their sources (the gathered token rows included)
  // are found once, so no k step waits on an index load.
  constexpr int kQ = (kTcBM * 8) / kTcThreads;
  static_assert(kTcBM == kTcBN, "one row set for both operands");
  const int cth = tid & 7, rth = tid >> 3;
  const uint16_t *a_src[kQ];
  const uint16_t *b_src[kQ];
  uint32_t a_ok = 0, b_ok = 0;
#pragma unroll
  for (int q = 0; q < kQ; ++q) {
    const int r = rth + 16 * q;
    a_src[q] = p.A;
    b_src[q] = p.B;
    if (r < rows) {
      const int g = row0 + r;
      const int arow = p.perm ? __ldg(p.perm + g) / p.ktop : g;
      a_src[q] = p.A + (size_t)arow * p.lda + cth * 8;
      a_ok |= 1u << q;
    }
    if (n0 + r < p.N) {
      const int n = n0 + r;
      const int brow = p.concat ? ((n & 1) ? p.N / 2 + (n >> 1) : (n >> 1)) : n;
      b_src[q] = p.B + ((size_t)e * p.N + brow) * p.K + cth * 8;
      b_ok |= 1u << q;
    }
  }
  auto load_stage = [&](int st, int k0) {
    unsigned char *As = base + (size_t)st * 2 * kTcTileBytes;
    unsigned char *Bs = As + kTcTileBytes;
#pragma unroll
    for (int q = 0; q < kQ; ++q) {
      const int r = rth + 16 * q;
      const bool ao = (a_ok >> q) & 1u, bo = (b_ok >> q) & 1u;
      cp_async16_zfill(smem_u32(As + tc_sw128(r, cth)), ao ? a_src[q] + k0 : p.A, ao ? 16u : 0u);
      cp_async16_zfill(smem_u32(Bs + tc_sw128(r, cth)), bo ? b_src[q] + k0 : p.B, bo ? 16u : 0u);
    }
  };

#pragma unroll
  for (int s = 0; s < kTcStages - 1; ++s) {
    if (s < KT) load_stage(s, s * kTcBK);
    cp_async_commit();
  }
  for (int kt = 0; kt < KT; ++kt) {
    cp_async_wait<kTcStages - 2>();
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // the tile is read by the tensor core
    __syncthreads();
    if (tid == 0) {
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const int st = kt % kTcStages;
      const uint32_t a_addr = smem_u32(base + (size_t)st * 2 * kTcTileBytes), b_addr = a_addr + kTcTileBytes;
#pragma unroll
      for (int kk = 0; kk < kTcBK / 16; ++kk) {
        const uint64_t da = tc_desc_sw128(a_addr + kk * 32), db = tc_desc_sw128(b_addr + kk * 32);
        const uint32_t acc = (kt > 0 || kk > 0) ? 1u : 0u;
        asm volatile(
            "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
            " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(tmem),
            "l"(da), "l"(db), "r"(kTcIdesc), "r"(acc)
            : "memory");
      }
      asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                       smem_u32(&mma_done[st]))
                   : "memory");
    }
    const int nk = kt + kTcStages - 1;
    if (nk < KT) {
      const int ns = nk % kTcStages;
      // stage ns was read by the MMAs of k step kt - 1: wait for them
      if (kt >= 1 && !s_abort && !tc_mbar_wait(&mma_done[ns], (uint32_t)((kt - 1) / kTcStages) & 1u)) {
        s_abort = 1;
        atomicCAS(err_flag, 0, 400);
      }
      load_stage(ns, nk * kTcBK);
    }
    cp_async_commit();
  }
  cp_async_wait<0>();
  if (!s_abort && !tc_mbar_wait(&mma_done[(KT - 1) % kTcStages], (uint32_t)((KT - 1) / kTcStages) & 1u)) {
    s_abort = 1;
    atomicCAS(err_flag, 0, 400);
  }
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");

  // epilogue: warp w holds accumulator rows 32w + lane
  const int r = warp * 32 + lane;
#pragma unroll 1
  for (int cc = 0; cc < kTcBN / 32; ++cc) {
    uint32_t v[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),
          "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),
          "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
        : "r"(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(cc * 32)));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
    const int c0 = n0 + cc * 32;
    if (r >= rows || c0 >= p.N) continue;  // N is a multiple of 64: a 32-column chunk is all in or all out
    const size_t prow = (size_t)(row0 + r);
    if (p.swiglu) {
      uint32_t o[8];
#pragma unroll
      for (int m = 0; m < 16; m += 2) {
        const float a0 = swiglu(__uint_as_float(v[2 * m]), __uint_as_float(v[2 * m + 1]), p.alpha, p.beta, p.limit);
        const float a1 =
            swiglu(__uint_as_float(v[2 * m + 2]), __uint_as_float(v[2 * m + 3]), p.alpha, p.beta, p.limit);
        o[m / 2] = f32_to_bf16_rne(a0) | (f32_to_bf16_rne(a1) << 16);
      }
      uint4 *dst = reinterpret_cast<uint4 *>(p.out_a + prow * (p.N / 2) + c0 / 2);
      dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
      dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
    } else {
      float4 *dst = reinterpret_cast<float4 *>(p.out_y + prow * p.N + c0);
#pragma unroll
      for (int q = 0; q < 8; ++q)
        dst[q] = make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]), __uint_as_float(v[4 * q + 2]),
                             __uint_as_float(v[4 * q + 3]));
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(128u) : "memory");
}

// xp[p] = x[perm_to_expanded[p] / k]: the token rows in expert order, 16
// bytes per thread and step, each row's copies coalesced.
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint16_t *__restrict__ x,
                                                          const int32_t *__restrict__ p2e, int R, int H, int k,
                                                          uint16_t *__restrict__ xp) {
  const int vpr = H / 8;  // 16-byte vectors per row
  const long long n = (long long)R * vpr;
  for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < n;
       idx += (long long)gridDim.x * blockDim.x) {
    const int pr = (int)(idx / vpr), v = (int)(idx - (long long)pr * vpr);
    const int t = __ldg(p2e + pr) / k;
    reinterpret_cast<uint4 *>(xp + (size_t)pr * H)[v] = __ldg(reinterpret_cast<const uint4 *>(x + (size_t)t * H) + v);
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
  // the shared-memory opt-in is a per-device attribute of the kernel
  static std::atomic<int> smem_set[kMaxDevices];
  const int dev = current_device();
  if (dev < 0) return cudaErrorInvalidDevice;
  if ((a.w1d || a.w2d) && !smem_set[dev].load(std::memory_order_acquire)) {
    cudaError_t err = cudaFuncSetAttribute(grouped_gemm_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmem);
    if (err != cudaSuccess) return err;
    smem_set[dev].store(1, std::memory_order_release);
  }
  int32_t *err_flag = a.err_flag;
  const int R = a.T * a.k;
  const int na_max = a.E < R ? a.E : R;
  const unsigned mtiles = (unsigned)((R + kTcBM - 1) / kTcBM + na_max);  // >= the sum over experts of ceil(rows / kTcBM)
  cudaError_t err;
  if (a.w1d) {
    GroupedGemm g1{};
    g1.A = a.x; g1.perm = a.p2e; g1.ktop = a.k; g1.lda = a.H;
    g1.B = a.w1d; g1.offsets = a.offsets; g1.E = a.E; g1.N = 2 * a.I; g1.K = a.H;
    g1.swiglu = 1; g1.concat = a.fusion == 2 ? 1 : 0;
    g1.out_a = a.act; g1.alpha = a.alpha; g1.beta = a.beta; g1.limit = a.limit;
    grouped_gemm_tc_kernel<<<dim3(mtiles, (unsigned)((g1.N + kTcBN - 1) / kTcBN)), kTcThreads, kTcSmem, stream>>>(
        g1, err_flag);
    err = cudaGetLastError();
  } else {
    const long long vecs = (long long)R * (a.H / 8);
    long long ggrid = (vecs + 255) / 256;
    if (ggrid > (long long)num_sms() * 8) ggrid = (long long)num_sms() * 8;
    gather_rows_kernel<<<(unsigned)ggrid, 256, 0, stream>>>(a.x, a.p2e, R, a.H, a.k, a.xp);
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    Fp4GemmArgs f{};
    f.mode = a.fusion == 2 ? 1 : 0;
    f.fmt = a.fmt; f.R = R; f.E = a.E; f.H = a.H; f.I = a.I;
    f.w = a.w1; f.s = a.s1k; f.gscale = a.g1;
    f.A = a.xp; f.offsets = a.offsets;
    f.out_a = a.act; f.alpha = a.alpha; f.beta = a.beta; f.limit = a.limit;
    f.err_flag = err_flag;
    err = launch_fp4_gemm(f, stream);
  }
  if (err != cudaSuccess) return err;
  stage_event(3, stream);
  if (a.w2d) {
    GroupedGemm g2{};
    g2.A = a.act; g2.perm = nullptr; g2.ktop = 1; g2.lda = a.I;
    g2.B = a.w2d; g2.offsets = a.offsets; g2.E = a.E; g2.N = a.H; g2.K = a.I;
    g2.swiglu = 0; g2.out_y = a.y;
    grouped_gemm_tc_kernel<<<dim3(mtiles, (unsigned)((g2.N + kTcBN - 1) / kTcBN)), kTcThreads, kTcSmem, stream>>>(
        g2, err_flag);
    err = cudaGetLastError();
  } else {
    Fp4GemmArgs f{};
    f.mode = 2;
    f.fmt = a.fmt; f.R = R; f.E = a.E; f.H = a.H; f.I = a.I;
    f.w = a.w2; f.s = a.s2k; f.gscale = a.g2;
    f.A = a.act; f.offsets = a.offsets;
    f.out_y = a.y;
    f.err_flag = err_flag;
    err = launch_fp4_gemm(f, stream);
  }
  if (err != cudaSuccess) return err;
  stage_event(4, stream);
  const long long work = (long long)a.T * (a.H / 2);
  long long grid = (work + 255) / 256;
  if (grid > (long long)num_sms() * 8) grid = (long long)num_sms() * 8;
  unpermute_kernel<<<(unsigned)grid, 256, 0, stream>>>(a.y, a.e2p, a.weights, a.T, a.H, a.k, a.out);
  err = cudaGetLastError();
  stage_event(5, stream);
  return err;
}

}  // namespace qmoe
