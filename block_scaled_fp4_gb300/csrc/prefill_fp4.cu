// Fused W4A16 grouped GEMM of the prefill path: the FP4 expert weights are
// decoded inside the GEMM, so no bf16 copy of them is written or read
// ("MoE and QMoE - CUDA Operator Documentation" §1 pipeline GEMM1 ->
// activation -> GEMM2, §4.3 and §9b for the E2M1 codes, the E4M3 / E8M0
// block scales and the fp32 global scale; the k-major block-scale layout
// [E, K/bs, N] of §9b.2).
//
// Product per tile (swapped operands): D[n][p] = sum_k W[k][n] * X[p][k] with
//  * M side (tcgen05 "A", 128 tensor-memory lanes) = 128 weight columns n,
//    decoded from the packed codes into shared memory as bf16, K-major with
//    the 128-byte swizzle.  The value written is the exact product
//    e2m1 * block scale (at most 6 significant bits, so exact in bf16); the
//    expert's global scale multiplies the fp32 accumulator in the epilogue;
//  * N side ("B") = the expert's token rows p in expert order, 16..160 of
//    them (one row chunk of one expert);
//  * fp32 accumulator in tensor memory, double-buffered (2 x 256 columns) so
//    that one tile's epilogue overlaps the next tile's MMAs.
// A row chunk is all of an expert's rows when they number <= 160, else an
// even split in multiples of 16: the MMA's N follows the expert's row count,
// so an expert with 130 rows costs 144 columns, not two 128-row tiles.
//
// Clusters of two CTAs (one per SM) take cluster tiles round-robin: a
// cluster tile is one row chunk and two consecutive column blocks, one per
// CTA, so the two CTAs need the same activation rows.  Roles in a CTA:
//  * MMA (one thread): tcgen05.mma kind::f16, M = 128, N = chunk rows,
//    K = 16, eight per 128-deep stage; commits release the decoded stage
//    locally and the activation stage in both CTAs (multicast commit);
//    the next stage's barriers are tested while this stage's MMAs issue;
//  * activation rows (one thread): 16-row tensor copies in the 128-byte
//    swizzle, each CTA copying half of a stage's boxes multicast to the
//    cluster, every CTA expecting the whole stage;
//  * packed codes and k-major scale rows (one warp, cp.async);
//  * decoders (eight warps): codes x scales -> bf16 M-side tile;
//  * epilogue (four warps, one per tensor-memory lane quadrant):
//    tcgen05.ld, x global scale, SwiGLU of the (gate, linear) pair and bf16
//    store of the activation (first GEMM), or fp32 store of the FC2 row.
// Every wait is bounded: on a timeout the CTA sets the device error flag,
// stops, waits (bounded) for its copies and MMAs in flight, meets its
// cluster and frees its tensor memory.
#include <atomic>

#include "decode_common.cuh"
#include "qmoe_common.cuh"

namespace qmoe {
namespace fg {

constexpr int kBM = 128;     // weight columns per tile (MMA M, tensor-memory lanes)
constexpr int kAtomK = 64;   // k of one 128-byte swizzled row of bf16 (a swizzle atom's depth)
constexpr int kBK = 128;     // k rows per stage: two atoms side by side, eight MMAs
constexpr int kHalves = kBK / kAtomK;
constexpr int kMaxN = 160;   // token rows per tile (MMA N)
constexpr int kAccCols = 256;  // tensor-memory columns between the two accumulator buffers
// Ring depths: the packed-weight ring covers HBM latency, the activation ring
// L2 latency, the decoded ring only the MMA's own latency.  A stage is 128
// deep so that the MMA thread's barrier tests and commits (each costs it
// about as much as an MMA issue) come once per eight MMAs.
constexpr int kPStages = 4, kBStages = 3, kAStages = 2;
constexpr int kBoxRows = 16;  // activation rows per tensor copy
// CTAs of a cluster share one row chunk (consecutive column blocks): each
// copies its share of the activation boxes, multicast to all of them.  Pairs
// measured faster than fours, of which only 36 fit on the device (144 SMs).
constexpr int kCluster = 2;
constexpr int kPLag = kPStages - 2;  // packed stages in flight before the copying warp publishes one
// Warp roles.  Warp w issues from scheduler w % 4, whose instruction cache
// it shares: the MMA warp's scheduler also runs only the two copy loops and
// one epilogue warp, the decoders' large unrolled loop runs on the other three.
//   scheduler 0: warp 0 MMA, 4 activation rows, 8 packed codes, 12 epilogue
//   schedulers 1-3: warps 1-3, 5-7, 9-10 decode, 11 idle, 13-15 epilogue
constexpr int kWarpMma = 0, kWarpRows = 4, kWarpCodes = 8, kWarpEpi0 = 12, kDecThreads = 256, kEpiThreads = 128;
constexpr int kThreads = 32 * kWarpEpi0 + kEpiThreads;  // 512
// decoder index of warp w (w % 4 != 0, w < kWarpEpi0): 0..8 in warp order
__host__ __device__ constexpr int dec_index(int w) { return (w / 4) * 3 + (w % 4) - 1; }
constexpr int kAHalf = kBM * kAtomK * 2;   // 16 KB: one atom-deep M-side tile
constexpr int kBHalf = kMaxN * kAtomK * 2; // 20 KB: one atom-deep N-side tile
constexpr int kATile = kHalves * kAHalf;
constexpr int kBTile = kHalves * kBHalf;
constexpr int kCodeBytes = kBK * kBM / 2;  // 8 KB: 128 k rows x 64 bytes
constexpr int kScaleBytes = (kBK / kNvfp4Block) * kBM;  // <= 8 block rows x 128 columns
constexpr int kPTile = kCodeBytes + kScaleBytes;
constexpr int kSmem = kAStages * kATile + kBStages * kBTile + kPStages * kPTile + 1024;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kWaitLimit = 1u << 22;
static_assert(kMaxN <= kAccCols && 2 * kAccCols <= (int)kTmemCols, "two accumulator buffers");
static_assert(kSmem <= 227 * 1024 - 4096, "stages fit in shared memory");
static_assert(kAHalf % 1024 == 0 && kBHalf % 1024 == 0, "atom tiles start on 1 KB swizzle boundaries");
static_assert(kEpiThreads == 128 && kWarpEpi0 % 4 == 0,
              "four epilogue warps: warp w reads tensor-memory lanes 32 (w % 4) ..");
static_assert(dec_index(kWarpEpi0 - 1) + 1 >= kDecThreads / 32, "enough decoder warps");

// MODE: 0 first GEMM, gate / linear interleaved (columns 2m, 2m + 1);
//       1 first GEMM, concatenated (columns m, I + m);
//       2 second GEMM.
struct Params {
  CUtensorMap tm_rows;     // bf16 activation rows in expert order [R][K], 128-byte swizzle, 64 x 16 boxes
  const uint8_t *codes;    // packed codes [E*K rows][N/2]
  const uint8_t *scales;   // k-major block scales [E*K/bs rows][N]
  const int32_t *offsets;  // [E + 1] first permuted row of each expert
  const float *gscale;     // [E] global scales, or null
  int E, K, N, I;          // expert weight: K x N; I: first GEMM's output width
  int ncb;                 // column blocks: I / 64 (first GEMM), ceil(N / 128) (second)
  int ncbg;                // column-block groups: ceil(ncb / kCluster)
  uint16_t *out_a;         // first GEMM: [R, I] bf16
  float *out_y;            // second GEMM: [R, N] fp32
  float alpha, beta, limit;
  int32_t *err_flag;
};

struct Bars {
  uint64_t pk_full[kPStages], pk_empty[kPStages];  // packed stage landed / read by the decoders
  uint64_t a_full[kAStages], a_empty[kAStages];    // decoded tile written / its MMAs done
  uint64_t b_full[kBStages], b_empty[kBStages];    // activation rows landed / their MMAs done

  uint64_t acc_full[2], acc_empty[2];              // accumulator buffers
  uint64_t drain;                                  // final MMA commit
};

struct Tile {
  int e, cb, r0, rows, nr;
};

// Cluster tile st = (chunk c of the expert-ordered chunk list, column-block
// group g); this CTA's column block is g * kCluster + its rank (>= ncb for
// the padding CTAs of a last, partial group: they copy and compute, but
// store nothing).
__device__ __forceinline__ Tile tile_at(const Params &p, const int *cpre, const int *offs, int st, int rank) {
  Tile T;
  const int c = st / p.ncbg;
  T.cb = (st - c * p.ncbg) * kCluster + rank;
  int lo = 0, hi = p.E;  // cpre[lo] <= c < cpre[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (cpre[mid] <= c) lo = mid;
    else hi = mid;
  }
  T.e = lo;
  const int n = offs[lo + 1] - offs[lo], nch = cpre[lo + 1] - cpre[lo], j = c - cpre[lo];
  const int cs = (((n + nch - 1) / nch) + 15) & ~15;
  T.r0 = offs[lo] + j * cs;
  T.rows = min(cs, n - j * cs);
  T.nr = (T.rows + 15) & ~15;
  return T;
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// 2-D tensor copy multicast to the CTAs of `mask`: each receives the box at
// the same shared-memory offset and a complete_tx on its mbarrier at `bar`'s
// offset.
__device__ __forceinline__ void tensor_g2s_2d_mc(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar,
                                                 uint16_t mask) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.multicast::cluster"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar)), "h"(mask)
      : "memory");
}

// Non-blocking test of a phase: issued early, its result is read only later,
// so that the check's latency overlaps other work.
__device__ __forceinline__ uint32_t mbar_test(uint64_t *bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done;
}

__device__ __forceinline__ bool wait_bounded(uint64_t *bar, uint32_t parity, volatile int *abort_s,
                                             int32_t *err_flag, int code) {
  for (uint32_t i = 0; i < kWaitLimit; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255u) == 255u && *abort_s) return false;
  }
  *abort_s = 1;
  atomicCAS(err_flag, 0, code);
  return false;
}

// Shared-memory matrix descriptor of a K-major, 128-byte-swizzled tile:
// start >> 4, leading byte offset 16 (unused with this swizzle), 1024 bytes
// between 8-row groups, descriptor version 1, swizzle mode 128 B.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// byte offset of 16-byte chunk c of row r in a K-major 128-byte-swizzled tile
__device__ __forceinline__ uint32_t sw128(int r, int c) { return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4)); }

__device__ __forceinline__ uint32_t bf16x2_of(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ float f16_lo(uint32_t h2) { return __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu))); }
__device__ __forceinline__ float f16_hi(uint32_t h2) { return __half2float(__ushort_as_half((unsigned short)(h2 >> 16))); }

// SwiGLU of one (gate, linear) pair with the fast exponential and reciprocal
// ("MoE and QMoE - CUDA Operator Documentation" §8: G = min(gate, limit),
// L = clamp(linear, -limit, limit), G * sigmoid(alpha * G) * (L + beta)).
__device__ __forceinline__ float swiglu_fast(float gate, float lin, float alpha, float beta, float limit) {
  const float G = fminf(gate, limit);
  const float L = fmaxf(fminf(lin, limit), -limit);
  return __fdividef(G, 1.0f + __expf(-alpha * G)) * (L + beta);
}

// ---- roles ----------------------------------------------------------------------

// Packed codes (64 k rows x 64 bytes) and k-major scale rows of a stage,
// copied by the 32 lanes of one warp with cp.async (the load/store path, so
// that the copy engine serves the activation rows alone); a stage is
// published kPLag stages later, once the lane's copies have landed.
template <int MODE, int FMT>
__device__ __forceinline__ void codes_role(const Params &p, const int *cpre, const int *offs, int nst, int rank,
                                           unsigned char *P_ring, Bars &B, volatile int *abort_s, int lane) {
  constexpr int BS = FMT == QMOE_NVFP4 ? kNvfp4Block : kMxfp4Block;
  constexpr int NSR = kBK / BS;  // scale block rows per stage
  const int KT = (p.K + kBK - 1) / kBK;
  const int rowb = p.N / 2;
  const int nclu = (int)gridDim.x / kCluster;
  uint32_t it = 0;
  bool ok = true;
  for (int st = (int)blockIdx.x / kCluster; st < nst && ok; st += nclu) {
    const Tile T = tile_at(p, cpre, offs, st, rank);
    const bool live = T.cb < p.ncb;
    for (int kt = 0; kt < KT; ++kt, ++it) {
      const int s = (int)(it % kPStages);
      const uint32_t u = it / kPStages;
      if (!wait_bounded(&B.pk_empty[s], (u & 1u) ^ 1u, abort_s, p.err_flag, 410)) {
        ok = false;
        break;
      }
      unsigned char *P = P_ring + (size_t)s * kPTile;
      const size_t row0 = (size_t)T.e * p.K + kt * kBK;
      const int krows = min(kBK, p.K - kt * kBK);  // 128, or 64 for a trailing half stage
      if (live) {
        // codes: krows x 64 bytes in chunks of 16 bytes, 16 per lane
#pragma unroll
        for (int c8 = 0; c8 < kBK * 4 / 32; ++c8) {
          const int ch = lane + 32 * c8, r = ch >> 2, cc = ch & 3;
          if (r >= krows) continue;
          if constexpr (MODE == 1) {
            const int piece = cc >> 1, c2 = cc & 1;
            const int xb = piece ? (p.I + 64 * T.cb) / 2 : 32 * T.cb;
            cp_async16(P + piece * (kCodeBytes / 2) + r * 32 + c2 * 16, p.codes + (row0 + r) * rowb + xb + c2 * 16);
          } else {
            const int xb = 64 * T.cb + cc * 16;
            if (xb < rowb) cp_async16(P + r * 64 + cc * 16, p.codes + (row0 + r) * rowb + xb);
          }
        }
        // scales: NSR rows x 128 bytes (those of the stage's krows)
        for (int c = lane; c < NSR * 8; c += 32) {
          const int r = c >> 3, cc = c & 7;
          if (r * BS >= krows) continue;
          const size_t srow = (size_t)T.e * (p.K / BS) + kt * NSR + r;
          if constexpr (MODE == 1) {
            const int piece = cc >> 2, c4 = cc & 3;
            const int xb = piece ? p.I + 64 * T.cb : 64 * T.cb;
            cp_async16(P + kCodeBytes + piece * NSR * 64 + r * 64 + c4 * 16, p.scales + srow * p.N + xb + c4 * 16);
          } else {
            const int xb = 128 * T.cb + cc * 16;
            if (xb < p.N) cp_async16(P + kCodeBytes + r * 128 + cc * 16, p.scales + srow * p.N + xb);
          }
        }
      }
      asm volatile("cp.async.commit_group;" ::: "memory");
      if (it >= (uint32_t)kPLag) {
        asm volatile("cp.async.wait_group %0;" ::"n"(kPLag) : "memory");
        mbar_arrive(&B.pk_full[(it - kPLag) % kPStages]);
      }
    }
  }
  asm volatile("cp.async.wait_group 0;" ::: "memory");
  if (ok) {
    const uint32_t n = it < (uint32_t)kPLag ? it : (uint32_t)kPLag;
    for (uint32_t d = n; d >= 1; --d) mbar_arrive(&B.pk_full[(it - d) % kPStages]);
  }
}

// Activation rows of a stage: nr rows x 64 k as tensor copies of 16 rows,
// written by the copy engine in the 128-byte-swizzled K-major layout the MMA
// descriptor reads (rows past the chunk's end are the next expert's or the
// copy's zero fill; their accumulator columns are never stored).  Every CTA
// of the cluster needs the same rows: CTA `rank` copies boxes rank,
// rank + kCluster, ... multicast to all, and expects the whole stage.
__device__ __forceinline__ void rows_role(const Params &p, const int *cpre, const int *offs, int nst, int rank,
                                          unsigned char *B_ring, Bars &B, volatile int *abort_s) {
  const int KT = (p.K + kBK - 1) / kBK;
  const int nclu = (int)gridDim.x / kCluster;
  const uint16_t all = (uint16_t)((1u << kCluster) - 1u);
  uint32_t it = 0;
  bool ok = true;
  for (int st = (int)blockIdx.x / kCluster; st < nst && ok; st += nclu) {
    const Tile T = tile_at(p, cpre, offs, st, rank);
    const int nbox = T.nr / kBoxRows;
    for (int kt = 0; kt < KT; ++kt, ++it) {
      const int s = (int)(it % kBStages);
      const uint32_t u = it / kBStages;
      // the stage is free in every CTA of the cluster (b_empty counts their MMA commits)
      if (!wait_bounded(&B.b_empty[s], (u & 1u) ^ 1u, abort_s, p.err_flag, 420)) {
        ok = false;
        break;
      }
      unsigned char *Bs = B_ring + (size_t)s * kBTile;
      // one atom-deep half after the other (a trailing stage may hold one half)
      const int nh = min(kHalves, (p.K - kt * kBK) / kAtomK);
      mbar_expect_tx(&B.b_full[s], (uint32_t)(nh * nbox * kBoxRows * kAtomK * 2));
      for (int h = 0; h < nh; ++h)
        for (int b = rank; b < nbox; b += kCluster)
          tensor_g2s_2d_mc(Bs + h * kBHalf + b * (kBoxRows * kAtomK * 2), &p.tm_rows, kt * kBK + h * kAtomK,
                           T.r0 + b * kBoxRows, &B.b_full[s], all);
    }
  }
  // before the CTA may leave: the copies into it have landed, and every CTA's
  // MMA commits for the last stages (remote arrivals on b_empty) are in
  const uint32_t n = it < (uint32_t)kBStages ? it : (uint32_t)kBStages;
  for (uint32_t d = 1; d <= n; ++d) {
    const uint32_t j = it - d;
    wait_bounded(&B.b_full[j % kBStages], (j / kBStages) & 1u, abort_s, p.err_flag, 421);
    wait_bounded(&B.b_empty[j % kBStages], (j / kBStages) & 1u, abort_s, p.err_flag, 422);
  }
}

// Decoder thread (w, kc, jh): column pairs 2jh, 2jh + 1 of column word w
// (tile columns 8w + 4jh .. 8w + 4jh + 3) over k rows 8kc..8kc+7 of each
// 64-deep half of the stage (its two swizzle-atom tiles).  Tile
// column n = 8w + j goes to M-side row 16j + w: a store phase of 8 lanes
// (w0..w0+7, one kc) then covers 8 distinct swizzle chunks.
template <int MODE, int FMT>
__device__ __forceinline__ void decoder_role(const Params &p, int my_steps, unsigned char *A_ring,
                                             const unsigned char *P_ring, Bars &B, volatile int *abort_s, int dt) {
  constexpr int BS = FMT == QMOE_NVFP4 ? kNvfp4Block : kMxfp4Block;
  constexpr int NSR = kBK / BS;
  const int lane = dt & 31, dw = dt >> 5;
  const int w = lane & 15, sw = lane >> 4, kc = 2 * (dw & 3) + sw, jh = dw >> 2;
  const int sr = (8 * kc) / BS;
  // byte offsets of this thread's code word in row 0 and of its 4 scales in
  // the first half; the second half is kAtomK code rows and kAtomK / BS
  // scale rows further on
  int code_off, pitch, sc_off, sc_pitch;
  if constexpr (MODE == 1) {
    code_off = (w >> 3) * (kCodeBytes / 2) + (w & 7) * 4;
    pitch = 32;
    sc_pitch = 64;
    sc_off = kCodeBytes + (w >> 3) * (NSR * 64) + sr * 64 + (w & 7) * 8 + 4 * jh;
  } else {
    code_off = w * 4;
    pitch = 64;
    sc_pitch = 128;
    sc_off = kCodeBytes + sr * 128 + w * 8 + 4 * jh;
  }
  for (int it = 0; it < my_steps; ++it) {
    const int s = it % kPStages;
    const uint32_t u = (uint32_t)it / kPStages;
    if (!wait_bounded(&B.pk_full[s], u & 1u, abort_s, p.err_flag, 430)) return;
    const unsigned char *P = P_ring + (size_t)s * kPTile;
    // half-warps read the two rows of a pair in opposite order: their row
    // parities differ, so the 32 loads hit 32 distinct banks
    uint32_t c[kHalves][8], svh[kHalves];
#pragma unroll
    for (int h = 0; h < kHalves; ++h) {
#pragma unroll
      for (int pr = 0; pr < 4; ++pr) {
        const int ra = h * kAtomK + 8 * kc + 2 * pr + sw, rb = h * kAtomK + 8 * kc + 2 * pr + (1 - sw);
        const uint32_t a = *reinterpret_cast<const uint32_t *>(P + code_off + ra * pitch);
        const uint32_t b = *reinterpret_cast<const uint32_t *>(P + code_off + rb * pitch);
        c[h][2 * pr] = sw ? b : a;
        c[h][2 * pr + 1] = sw ? a : b;
      }
      svh[h] = *reinterpret_cast<const uint32_t *>(P + sc_off + h * (kAtomK / BS) * sc_pitch);
    }
    mbar_arrive(&B.pk_empty[s]);
    const int sa = it % kAStages;
    const uint32_t ua = (uint32_t)it / kAStages;
    if (!wait_bounded(&B.a_empty[sa], (ua & 1u) ^ 1u, abort_s, p.err_flag, 431)) return;
#pragma unroll
    for (int h = 0; h < kHalves; ++h) {
    unsigned char *As = A_ring + (size_t)sa * kATile + h * kAHalf;
    const uint32_t sv = svh[h];
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int jj = 2 * jh + q;  // column pair of the word
      float lo[8], hi[8];
      if constexpr (FMT == QMOE_NVFP4) {
        const uint32_t sh = e4m3x2_to_f16x2((sv >> (16 * q)) & 0xFFFFu);
        const uint16_t s_lo = (uint16_t)(sh & 0xFFFFu), s_hi = (uint16_t)(sh >> 16);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint32_t v = e2m1x2_to_f16x2(c[h][i] >> (8 * jj));
          lo[i] = fma_f16_f32((uint16_t)(v & 0xFFFFu), s_lo, -0.0f);
          hi[i] = fma_f16_f32((uint16_t)(v >> 16), s_hi, -0.0f);
        }
      } else {
        const uint32_t sb = sv >> (16 * q);
        const float f_lo = e8m0_to_f32(sb & 0xFFu), f_hi = e8m0_to_f32((sb >> 8) & 0xFFu);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint32_t v = e2m1x2_to_f16x2(c[h][i] >> (8 * jj));
          lo[i] = f16_lo(v) * f_lo;
          hi[i] = f16_hi(v) * f_hi;
        }
      }
      const int ar0 = 16 * (2 * jj) + w, ar1 = ar0 + 16;
      *reinterpret_cast<uint4 *>(As + sw128(ar0, kc)) =
          make_uint4(bf16x2_of(lo[0], lo[1]), bf16x2_of(lo[2], lo[3]), bf16x2_of(lo[4], lo[5]), bf16x2_of(lo[6], lo[7]));
      *reinterpret_cast<uint4 *>(As + sw128(ar1, kc)) =
          make_uint4(bf16x2_of(hi[0], hi[1]), bf16x2_of(hi[2], hi[3]), bf16x2_of(hi[4], hi[5]), bf16x2_of(hi[6], hi[7]));
    }
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    mbar_arrive(&B.a_full[sa]);
  }
}

__device__ __forceinline__ void mma_commit(uint64_t *bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
               : "memory");
}

__device__ __forceinline__ void mma_role(const Params &p, const int *cpre, const int *offs, int nst, int rank,
                                         const unsigned char *A_ring, const unsigned char *B_ring, Bars &B,
                                         uint32_t tmem, volatile int *abort_s) {
  const int KT = (p.K + kBK - 1) / kBK;
  uint32_t it = 0, tl = 0;
  bool ok = true;
  const int nclu = (int)gridDim.x / kCluster;
  const uint16_t all = (uint16_t)((1u << kCluster) - 1u);
  bool ready = false;  // the next stage's barriers were found complete
  for (int st = (int)blockIdx.x / kCluster; st < nst && ok; st += nclu, ++tl) {
    const Tile T = tile_at(p, cpre, offs, st, rank);
    const uint32_t ab = tl & 1u, ua = tl >> 1;
    if (!wait_bounded(&B.acc_empty[ab], (ua & 1u) ^ 1u, abort_s, p.err_flag, 440)) break;
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t d = tmem + ab * (uint32_t)kAccCols;
    // fp32 accumulator, bf16 A and B, both K-major, N >> 3 at bit 17, M >> 4 at bit 24
    const uint32_t idesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(T.nr >> 3) << 17) |
                           ((uint32_t)(kBM >> 4) << 24);
    for (int kt = 0; kt < KT; ++kt, ++it) {
      const int sa = (int)(it % kAStages), sb = (int)(it % kBStages);
      // the test of this stage's barriers was issued during the previous
      // stage's MMAs; wait only if it found them incomplete
      if (!ready && (!wait_bounded(&B.a_full[sa], (it / kAStages) & 1u, abort_s, p.err_flag, 441) ||
                     !wait_bounded(&B.b_full[sb], (it / kBStages) & 1u, abort_s, p.err_flag, 442))) {
        ok = false;
        break;
      }
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const uint32_t nx = it + 1;
      const uint32_t ta = mbar_test(&B.a_full[nx % kAStages], (nx / kAStages) & 1u);
      const uint32_t tb = mbar_test(&B.b_full[nx % kBStages], (nx / kBStages) & 1u);
      const uint32_t a_addr = smem_addr(A_ring + (size_t)sa * kATile), b_addr = smem_addr(B_ring + (size_t)sb * kBTile);
      const int nkk = min(kBK, p.K - kt * kBK) / 16;  // 8, or 4 in a trailing half stage
#pragma unroll
      for (int kk = 0; kk < kBK / 16; ++kk) {
        if (kk >= nkk) break;
        // 16-deep slice kk: atom tile kk / 4, 32 bytes per slice within it
        const int h = kk / (kAtomK / 16), ks = kk % (kAtomK / 16);
        const uint64_t da = desc_sw128(a_addr + h * kAHalf + ks * 32), db = desc_sw128(b_addr + h * kBHalf + ks * 32);
        const uint32_t acc = (kt > 0 || kk > 0) ? 1u : 0u;
        asm volatile(
            "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
            " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d),
            "l"(da), "l"(db), "r"(idesc), "r"(acc)
            : "memory");
      }
      mma_commit(&B.a_empty[sa]);
      // the activation stage is free for the copies once every CTA's MMAs are done with it
      asm volatile(
          "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
              smem_addr(&B.b_empty[sb])),
          "h"(all)
          : "memory");
      ready = (ta & tb) != 0u;
    }
    if (!ok) break;
    mma_commit(&B.acc_full[ab]);
  }
  // every MMA issued above has completed before the tensor memory is freed
  mma_commit(&B.drain);
  wait_bounded(&B.drain, 0u, abort_s, p.err_flag, 443);
}

// Epilogue thread: tensor-memory lane 32q + l = M-side row 16j + w, i.e. tile
// column n = 8w + j with w = l & 15, j = 2q + (l >> 4).
template <int MODE>
__device__ __forceinline__ void epilogue_role(const Params &p, const int *cpre, const int *offs, int nst, int rank,
                                              Bars &B, uint32_t tmem, volatile int *abort_s, int warp) {
  const int q = warp & 3, lane = (int)lane_id();
  const int w = lane & 15, j = 2 * q + (lane >> 4), n = 8 * w + j;
  // first GEMM: (gate, linear) partners are lanes l and l ^ 16 (interleaved:
  // j even / odd, same w) or l and l ^ 8 (concatenated: w < 8 / >= 8, same
  // j).  Of rows 2a and 2a + 1 the gate lane finishes row 2a, the linear
  // lane row 2a + 1, each with the value the other sends it.
  constexpr int kX = MODE == 0 ? 16 : 8;
  const bool gate = MODE == 0 ? (lane < 16) : (w < 8);
  const int m_in = MODE == 0 ? 4 * w + q : 8 * (w & 7) + j;  // output column of the pair within the tile
  uint32_t tl = 0;
  const int nclu = (int)gridDim.x / kCluster;
  for (int st = (int)blockIdx.x / kCluster; st < nst; st += nclu, ++tl) {
    const Tile T = tile_at(p, cpre, offs, st, rank);
    const uint32_t ab = tl & 1u, ua = tl >> 1;
    if (!wait_bounded(&B.acc_full[ab], ua & 1u, abort_s, p.err_flag, 450)) return;
    const bool live = T.cb < p.ncb;
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const float g = p.gscale ? __ldg(p.gscale + T.e) : 1.0f;
    const uint32_t tbase = tmem + ((uint32_t)(32 * q) << 16) + ab * (uint32_t)kAccCols;
    for (int cc = 0; live && cc * 32 < T.nr; ++cc) {
      uint32_t v[32];
      asm volatile(
          "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
          "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
          : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
            "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),
            "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),
            "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
          : "r"(tbase + (uint32_t)(cc * 32)));
      asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
      const int rbase = cc * 32;
      if constexpr (MODE == 2) {
        const int h = 128 * T.cb + n;
        if (h < p.N) {
          float *dst = p.out_y + (size_t)(T.r0 + rbase) * p.N + h;
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (rbase + i < T.rows) dst[(size_t)i * p.N] = __uint_as_float(v[i]) * g;
        }
      } else {
        const int r_odd = gate ? 0 : 1;  // which row of each pair this lane finishes
        uint16_t *dst = p.out_a + (size_t)(T.r0 + rbase + r_odd) * p.I + 64 * T.cb + m_in;
#pragma unroll
        for (int a = 0; a < 16; ++a) {
          const float v0 = __uint_as_float(v[2 * a]) * g, v1 = __uint_as_float(v[2 * a + 1]) * g;
          // gate lane sends its row-(2a+1) gate, linear lane its row-2a linear
          const float got = __shfl_xor_sync(0xFFFFFFFFu, gate ? v1 : v0, kX);
          const float gv = gate ? v0 : got, lv = gate ? got : v1;
          if (rbase + 2 * a + r_odd < T.rows)
            dst[(size_t)(2 * a) * p.I] = (uint16_t)f32_to_bf16_rne(swiglu_fast(gv, lv, p.alpha, p.beta, p.limit));
        }
      }
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    mbar_arrive(&B.acc_empty[ab]);
  }
}

template <int MODE, int FMT>
__global__ void __launch_bounds__(kThreads, 1) fp4_grouped_gemm_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(1024) unsigned char dsm[];
  __shared__ Bars B;
  __shared__ uint32_t tmem_s;
  __shared__ int cpre[kMaxExperts + 1], offs[kMaxExperts + 1];
  __shared__ volatile int abort_s;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  unsigned char *base = dsm + ((1024u - (smem_addr(dsm) & 1023u)) & 1023u);
  unsigned char *A_ring = base;
  unsigned char *B_ring = A_ring + kAStages * kATile;
  unsigned char *P_ring = B_ring + kBStages * kBTile;

  if (warp == kWarpMma) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(&tmem_s)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  } else if (warp == kWarpCodes && lane == 0) {
    for (int i = 0; i < kPStages; ++i) {
      mbar_init(&B.pk_full[i], 32);
      mbar_init(&B.pk_empty[i], kDecThreads);
    }
    for (int i = 0; i < kAStages; ++i) {
      mbar_init(&B.a_full[i], kDecThreads);
      mbar_init(&B.a_empty[i], 1);
    }
    for (int i = 0; i < kBStages; ++i) {
      mbar_init(&B.b_full[i], 1);
      mbar_init(&B.b_empty[i], kCluster);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&B.acc_full[i], 1);
      mbar_init(&B.acc_empty[i], kEpiThreads);
    }
    mbar_init(&B.drain, 1);
    mbar_fence_init();
    abort_s = 0;
  } else if (warp == kWarpRows) {  // chunks per expert and their prefix (E <= 256)
    const int per = (p.E + 31) / 32;
    int sum = 0;
    for (int q = 0; q < per; ++q) {
      const int e = lane * per + q;
      if (e <= p.E) offs[e] = __ldg(p.offsets + e);
      if (e < p.E) sum += (__ldg(p.offsets + e + 1) - __ldg(p.offsets + e) + kMaxN - 1) / kMaxN;
    }
    if (lane == 31 && per * 32 == p.E) offs[p.E] = __ldg(p.offsets + p.E);
    int incl = sum;
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
      const int v = __shfl_up_sync(0xFFFFFFFFu, incl, m);
      if (lane >= m) incl += v;
    }
    int run = incl - sum;
    for (int q = 0; q < per; ++q) {
      const int e = lane * per + q;
      if (e < p.E) {
        cpre[e] = run;
        run += (__ldg(p.offsets + e + 1) - __ldg(p.offsets + e) + kMaxN - 1) / kMaxN;
      }
    }
    if (lane == 31) cpre[p.E] = incl;
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  // every CTA's barriers are initialised before a peer's multicast signals them
  cluster_sync();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = tmem_s;
  const int rank = (int)cluster_rank();
  const int nst = cpre[p.E] * p.ncbg;

  if (warp == kWarpMma) {
    if (lane == 0) mma_role(p, cpre, offs, nst, rank, A_ring, B_ring, B, tmem, &abort_s);
    __syncwarp();
  } else if (warp == kWarpCodes) {
    codes_role<MODE, FMT>(p, cpre, offs, nst, rank, P_ring, B, &abort_s, lane);
  } else if (warp == kWarpRows) {
    if (lane == 0) rows_role(p, cpre, offs, nst, rank, B_ring, B, &abort_s);
    __syncwarp();
  } else if (warp < kWarpEpi0) {
    const int di = dec_index(warp);
    if (di < kDecThreads / 32) {
      const int ci = (int)blockIdx.x / kCluster, nclu = (int)gridDim.x / kCluster;
      const int mine = ci < nst ? (nst - ci + nclu - 1) / nclu : 0;
      decoder_role<MODE, FMT>(p, mine * ((p.K + kBK - 1) / kBK), A_ring, P_ring, B, &abort_s, 32 * di + lane);
    }
  } else {
    epilogue_role<MODE>(p, cpre, offs, nst, rank, B, tmem, &abort_s, warp);
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  // no CTA leaves while a peer may still multicast into it or signal its barriers
  cluster_sync();
  if (warp == kWarpMma) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// A 2-D byte array [rows][cols] (row pitch = cols) as a tensor map with a
// box of box_cols x box_rows.
static cudaError_t encode_fn(EncodeTiledFn *out) {
  static std::atomic<EncodeTiledFn> fn{nullptr};
  EncodeTiledFn f = fn.load(std::memory_order_acquire);
  if (!f) {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q);
    if (err != cudaSuccess || q != cudaDriverEntryPointSuccess || !ptr) {
      set_error("cuTensorMapEncodeTiled is not available");
      return err != cudaSuccess ? err : cudaErrorNotSupported;
    }
    f = reinterpret_cast<EncodeTiledFn>(ptr);
    fn.store(f, std::memory_order_release);
  }
  *out = f;
  return cudaSuccess;
}

// bf16 rows [rows][cols] as a tensor map with 64 x kBoxRows boxes in the
// 128-byte swizzle (16-byte chunk c of box row r at chunk c ^ (r & 7)).
static cudaError_t encode_rows_sw128(CUtensorMap *m, const void *base, uint64_t cols, uint64_t rows) {
  EncodeTiledFn f = nullptr;
  cudaError_t err = encode_fn(&f);
  if (err != cudaSuccess) return err;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kAtomK, (cuuint32_t)kBoxRows};
  const cuuint32_t es[2] = {1, 1};
  const CUresult r = f(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, es,
                       CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_error("cuTensorMapEncodeTiled failed (%d)", (int)r);
    return cudaErrorInvalidValue;
  }
  return cudaSuccess;
}

// Launch as clusters of kCluster CTAs, one CTA per SM, as many clusters as
// fit on the device at once (at most one per cluster tile).
template <int MODE, int FMT>
static cudaError_t launch_mode(const Params &p, long long max_clusters, cudaStream_t stream) {
  static std::atomic<int> fit[kMaxDevices];  // clusters resident at once, per device (0: not yet known)
  const int dev = current_device();
  if (dev < 0) return cudaErrorInvalidDevice;
  auto kfn = fp4_grouped_gemm_kernel<MODE, FMT>;
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kCluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = fit[dev].load(std::memory_order_acquire);
  if (n == 0) {
    cudaError_t err = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (err != cudaSuccess) return err;
    cfg.gridDim = dim3(kCluster * (unsigned)(num_sms() / kCluster), 1, 1);
    err = cudaOccupancyMaxActiveClusters(&n, kfn, &cfg);
    if (err != cudaSuccess) return err;
    if (n < 1) {
      set_error("the fused prefill GEMM's %d-CTA clusters do not fit on this device", kCluster);
      return cudaErrorInvalidConfiguration;
    }
    fit[dev].store(n, std::memory_order_release);
  }
  const long long clusters = max_clusters < n ? max_clusters : n;
  cfg.gridDim = dim3((unsigned)(clusters * kCluster), 1, 1);
  return cudaLaunchKernelEx(&cfg, kfn, p);
}

}  // namespace fg

cudaError_t launch_fp4_gemm(const Fp4GemmArgs &a, cudaStream_t stream) {
  using namespace fg;
  Params p{};
  const bool first = a.mode != 2;
  const int N = first ? 2 * a.I : a.H, K = first ? a.H : a.I;
  const int R = a.R;
  if (R <= 0) return cudaSuccess;
  p.codes = a.w; p.scales = a.s;
  p.offsets = a.offsets; p.gscale = a.gscale;
  p.E = a.E; p.K = K; p.N = N; p.I = a.I;
  p.ncb = first ? a.I / 64 : (a.H + kBM - 1) / kBM;
  p.ncbg = (p.ncb + kCluster - 1) / kCluster;
  p.out_a = a.out_a; p.out_y = a.out_y;
  p.alpha = a.alpha; p.beta = a.beta; p.limit = a.limit;
  p.err_flag = a.err_flag;
  cudaError_t err = encode_rows_sw128(&p.tm_rows, a.A, (uint64_t)K, (uint64_t)R);
  if (err != cudaSuccess) return err;
  // cluster tiles <= (sum over experts of ceil(rows / kMaxN)) * column-block groups
  const long long chunks = (long long)R / kMaxN + (a.E < R ? a.E : R) + 1;
  const long long max_clusters = chunks * p.ncbg;
  const bool nv = a.fmt == QMOE_NVFP4;
  switch (a.mode) {
    case 0: return nv ? launch_mode<0, QMOE_NVFP4>(p, max_clusters, stream) : launch_mode<0, QMOE_MXFP4>(p, max_clusters, stream);
    case 1: return nv ? launch_mode<1, QMOE_NVFP4>(p, max_clusters, stream) : launch_mode<1, QMOE_MXFP4>(p, max_clusters, stream);
    default: return nv ? launch_mode<2, QMOE_NVFP4>(p, max_clusters, stream) : launch_mode<2, QMOE_MXFP4>(p, max_clusters, stream);
  }
}

}  // namespace qmoe
