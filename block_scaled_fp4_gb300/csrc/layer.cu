// Decode path of the FP4 MoE layer in one persistent kernel: top-k softmax
// routing and the permute maps, FC1 GEMV with SwiGLU, FC2 GEMV and the
// weighted un-permute, with the E2M1 weights dequantised in registers.
//
// Prior art on the pages ("[CUDA] Speed up the NVFP4 QMoE decode GEMV and
// enable it for MTP verify", PR #31159; operator doc §9b.2/§9b.3): coalesced
// weight and scale streams, weight loads batched ahead of their decode, a
// table-free E2M1 decode, the block scale applied to a per-block partial sum
// instead of to every weight, fp32 accumulation for bf16 activations, and a
// 64-expanded-row window.  Design here (sm_103a, one CTA per SM):
//  * every CTA routes the (at most 64) expanded rows itself with the routing
//    kernel's warp top-k and a one-warp stable ranking, so all CTAs hold
//    identical maps and no separate launch sits between the call and the
//    weight stream;
//  * work unit = 16*RGS k rows x NT columns of one active expert's weights
//    (about 32 KB).  The units of all active experts are laid end to end
//    (expert slot, column tile, k) and split over the CTAs by cost
//    ("stream-K"): every CTA streams about the same bytes whatever the number
//    of rows each expert received.  A CTA's consecutive units of one
//    (expert, tile) form a segment, which it reduces to a partial sum;
//  * one warp issues the bulk async copies (cp.async.bulk, completion counted
//    on an mbarrier) of the CTA's FC1 units and then, without waiting for FC1
//    to finish anywhere, of its FC2 units into a 3- or 4-slot ring.  With
//    k-major block scales ([E, K/bs, N]) a unit's scale rows travel in its
//    slot; with the [E, N, K/bs] layout, windows of 16 blocks are 2-D tensor
//    copies transposed per warp (NVFP4) or byte loads;
//  * a second warp copies each pass's activation rows with cp.async (the
//    load/store path, so they do not queue behind the weight stream);
//  * 16 consumer warps: thread (w, rg) owns column word w (8 columns) of
//    k-group rg (16 rows) of a unit, decodes with the hardware
//    cvt.rn.f16x2.e2m1x2 and multiplies with fma.rn.f32.f16 (fp16 operands,
//    exact product, fp32 accumulator); the 16-row partial is multiplied once
//    by its block scale (NVFP4: the E4M3 value from the hardware conversion
//    cvt.rn.f16x2.e4m3x2, exact; MXFP4: 2^(b-127) by bit placement);
//  * activations are staged in fp16 after an exact power-of-two rescale per
//    row (largest |x| in [2^14, 2^15)), so every finite bf16 activation is
//    exact in fp16; the rescale is undone on the fp32 partial;
//  * partial sums are reduced over row groups with warp shuffles and written
//    to global memory (fp32).  After a grid barrier, FC2 forms its bf16
//    activations a = SwiGLU(g1 * sum of FC1 partials) for the k range it
//    needs; after a second grid barrier, out[t] = bf16(sum_j w[t][j] * g2 *
//    sum of FC2 partials of (t, j)).  All sums run in a fixed order, so the
//    result is deterministic;
//  * the kernel is launched cooperatively (all CTAs resident, so the grid
//    barriers cannot deadlock).  Its barrier counters live in the workspace
//    header; the last CTA out returns them to zero, so a call on a workspace
//    whose header is known to be zero needs no reset and is launched with
//    programmatic dependent launch right behind the previous kernel;
//  * every wait is bounded: a wait that gives up sets the device error flag
//    meta[1] and the CTA carries on without waiting again, so no CTA hangs.
#include <cuda.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <atomic>

#include "decode_common.cuh"

namespace qmoe {

constexpr int kCons = 512;                 // consumer threads
constexpr int kConsWarps = kCons / 32;
constexpr int kLayerThreads = kCons + 64;  // + the weight-copy warp + the activation/scale-copy warp
constexpr int kWarpW = kConsWarps;
constexpr int kWarpS = kConsWarps + 1;
constexpr int kRingMax = 4;                // weight ring slots (LayerPlan::ring: 4 when shared memory allows, else 3)
constexpr int kTmaWB = 16;                 // blocks per scale window copied by the tensor unit
constexpr int kTmaMaxNT = 1024;            // so that a window is at most 16 KB
constexpr int kMaxWinBytes = 16 * 1024;
constexpr int kSmemOptin = 232448;         // shared memory per block (opt-in) on sm_100 / sm_103
constexpr int kMaxSegs = 32;               // segments of one FC in one CTA
constexpr int kMaxCtas = 256;              // grid size (one CTA per SM)
constexpr int kXsK = 512;                  // activations staged per row at a time (per warp)
constexpr int kRowsMax = 1;                // rows per pass: a row of an expert is one pass over its units
constexpr int kXrawSlot = kRowsMax * kXsK * 2;  // bytes of one raw (bf16) activation slot
constexpr int kXrawBytes = 16 * 1024;            // FC1: two slots at the start; FC2: pre-staged activations
constexpr int kXwBytes = kRowsMax * kXsK * 2;    // one warp's fp16 activation window
constexpr int kMaxSlots = 64;
constexpr int kMaxTiles = 16;
constexpr int kMaxPairs = kMaxSlots * kMaxTiles;
constexpr uint32_t kWaitLimit = 1u << 22;
constexpr uint32_t kSpinLimit = 1u << 24;
static_assert(2 * kXrawSlot <= kXrawBytes, "two raw activation slots");

// Consumer threads only (the copy and scale warps never take part).
__device__ __forceinline__ void cons_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kCons) : "memory"); }

// v_i byte q = scale of column i at block q  ->  row q of dst = the 4 columns' bytes
__device__ __forceinline__ void store_tile4x4(uint32_t v0, uint32_t v1, uint32_t v2, uint32_t v3, uint8_t *dst,
                                              int stride, int rows) {
  const uint32_t t01lo = __byte_perm(v0, v1, 0x5140), t01hi = __byte_perm(v0, v1, 0x7362);
  const uint32_t t23lo = __byte_perm(v2, v3, 0x5140), t23hi = __byte_perm(v2, v3, 0x7362);
  const uint32_t rr[4] = {__byte_perm(t01lo, t23lo, 0x5410), __byte_perm(t01lo, t23lo, 0x7632),
                          __byte_perm(t01hi, t23hi, 0x5410), __byte_perm(t01hi, t23hi, 0x7632)};
#pragma unroll
  for (int q = 0; q < 4; ++q)
    if (q < rows) *reinterpret_cast<uint32_t *>(dst + (size_t)q * stride) = rr[q];
}

// ---- work geometry ------------------------------------------------------------------

// Work split: the units of FC f, in (expert slot, column tile, k) order, are
// cut into gridDim.x ranges of about equal cost; CTA c gets units
// [bnd[f][c], bnd[f][c + 1]).  Costs are in 1/64 of one unit decoded for one
// row.  A CTA spends, on each segment (its units of one pair) of an r-row
// expert, r * (pass start + 64 * units): every row is one pass over the
// units.  Every CTA pays at least one segment; the CTA that crosses into a
// new pair pays one more, so each pair start is charged r * pass_cost.  The
// per-unit cost of an r-row expert, P.ucost[r - 1] (host table), is what makes
// a CTA inside such a pair take as long as one inside a one-row pair despite
// its r pass starts.
__device__ __forceinline__ int unit_cost(const FcPlan &P, int rows) {
  return P.ucost[min(rows, kCostRows) - 1];
}
__device__ __forceinline__ int pair_cost(const FcPlan &P, int rows) {
  return rows * P.pass_cost + P.ku * unit_cost(P, rows);
}

struct FcWork {
  int lo, hi;
};
// CTA holding unit u: the largest c with bnd[c] <= u (empty ranges skipped).
__device__ __forceinline__ int cta_of(const int *bnd, int u) {
  int lo = 0, hi = (int)gridDim.x - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (bnd[mid] <= u) lo = mid; else hi = mid - 1;
  }
  return lo;
}
// Scale window holding the blocks of unit j (a unit never straddles two).
template <int FMT>
__device__ __forceinline__ int unit_window(const FcPlan &P, int j) {
  constexpr int BS = FMT == QMOE_NVFP4 ? kNvfp4Block : kMxfp4Block;
  return ((j * P.RGS * 16) / BS) / P.WB;
}
__device__ __forceinline__ int unit_rows(const FcPlan &P, int j) { return min(16 * P.RGS, P.K - j * 16 * P.RGS); }

// A CTA's consecutive units of one (expert slot, column tile) pair.
struct Seg {
  int pair, a, t, j0, j1, wid0, wid1;
  int dst;  // offset (floats) of this CTA's partial rows of the pair (set with the partial-sum bases)
};

struct Shared {
  uint64_t full[kRingMax], empty[kRingMax];  // weight ring
  uint64_t wfull[2], wempty[2];        // scale-window staging
  uint64_t xfull[2], xempty[2];        // raw FC1 activation slots
  uint64_t gsready, smallfirst, basesready;
  int4 slot[kMaxSlots];                // {e, row0, nrows, -}
  float gs[2][kMaxSlots];              // global scales per slot (1 for MXFP4)
  int base[2][kMaxPairs + 1];          // partial-sum offsets (floats) per (slot, tile) pair
  Seg seg[2][kMaxSegs];
  int nseg[2];
  int bnd[2][kMaxCtas + 1];            // work split (units)
  short pcnt[2][kMaxPairs];            // partial-sum slots (CTAs holding units) of each pair
  short busy[2][kMaxCtas + 1];         // CTAs holding units among [0, c)
  int scum[2][kMaxSlots + 1];          // cost prefix over expert slots
  int row2slot[kMaxSlots];
  int row_tok[kMaxSlots];              // token of each permuted row
  // routing (computed by every CTA for itself): expert and weight of each
  // expanded row t * k + j and the permute maps
  int r_ids[kMaxSlots];
  float r_w[kMaxSlots];
  int r_e2p[kMaxSlots];
  int r_p2e[kMaxSlots];
  uint32_t wmax[kConsWarps];
  int na;
  int abort;
  int fc2_pre;                         // FC2 activations pre-staged in the raw buffer
};

__device__ __forceinline__ FcWork fc_work(const Shared &S, int f) {
  return FcWork{S.bnd[f][blockIdx.x], S.bnd[f][blockIdx.x + 1]};
}
// The CTAs holding the first and the last unit of (expert slot, tile) pair p.
__device__ __forceinline__ int first_cta(const Shared &S, const FcPlan &P, int f, int p) {
  return cta_of(S.bnd[f], p * P.ku);
}
__device__ __forceinline__ int last_cta(const Shared &S, const FcPlan &P, int f, int p) {
  return cta_of(S.bnd[f], p * P.ku + P.ku - 1);
}
// CTAs in [c0, c1) that hold at least one unit.  The partial-sum slots of a
// pair are numbered by these only: a CTA with an empty range writes nothing.
__device__ __forceinline__ int busy_ctas(const Shared &S, int f, int c0, int c1) {
  return S.busy[f][c1] - S.busy[f][c0];
}

__device__ __forceinline__ bool wait_bar(Shared &S, const LayerArgs &g, uint64_t *bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;  // the usual case: no abort-flag read
  const uint32_t limit = *(volatile int *)&S.abort ? 64u : kWaitLimit;
  for (uint32_t i = 0; i < limit; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  *(volatile int *)&S.abort = 1;
  // the flag keeps the first failure: 100 + the barrier's index in the shared block
  atomicCAS(g.meta + 1, 0, 100 + (int)(bar - reinterpret_cast<uint64_t *>(&S)));
  return false;
}

__device__ void grid_barrier(Shared &S, const LayerArgs &g, int32_t *ctr) {
  cons_sync();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(ctr, 1);
    const uint32_t limit = *(volatile int *)&S.abort ? 1024u : kSpinLimit;
    for (uint32_t i = 0; ld_acquire(ctr) < (int)gridDim.x; ++i) {
      if (i >= limit) {
        *(volatile int *)&S.abort = 1;
        atomicCAS(g.meta + 1, 0, 200 + (int)(ctr - g.meta));  // 202, 203: the grid barriers
        break;
      }
      __nanosleep(64);
    }
  }
  cons_sync();
}

// Called by each CTA's barrier thread after its last poll of a barrier
// counter (those polls are acquire loads, so they stay before it): the last
// CTA to count itself out returns both barrier counters and this counter to
// zero, so the next call on the workspace starts from zero without a reset.
__device__ void leave_counters(const LayerArgs &g) {
  if (atomicAdd(g.meta + 4, 1) == (int)gridDim.x - 1) {
    atomicExch(g.meta + 2, 0);
    atomicExch(g.meta + 3, 0);
    atomicExch(g.meta + 4, 0);
  }
}

// ---- set-up ----------------------------------------------------------------------------

// This CTA's segments of FC f (one warp, one lane per segment): the pairs
// its unit range [lo, hi) touches, each cut to that range.
template <int FMT>
__device__ void build_segments(Shared &S, const LayerArgs &g, const FcPlan &P, int f) {
  const int lane = (int)lane_id();
  const FcWork W = fc_work(S, f);
  const int p0 = W.lo / P.ku, n = W.lo < W.hi ? (W.hi - 1) / P.ku - p0 + 1 : 0;
  if (n > kMaxSegs) {  // the host bounds this; report rather than drop work
    if (lane == 0) {
      *(volatile int *)&S.abort = 1;
      atomicCAS(g.meta + 1, 0, 300);  // more segments than the kernel holds
    }
  }
  const int nseg = min(n, kMaxSegs);
  if (lane < nseg) {
    const int pair = p0 + lane;
    Seg sg;
    sg.pair = pair;
    sg.a = pair / P.ct;
    sg.t = pair - sg.a * P.ct;
    sg.j0 = max(W.lo, pair * P.ku) - pair * P.ku;
    sg.j1 = min(W.hi, (pair + 1) * P.ku) - pair * P.ku;
    sg.wid0 = unit_window<FMT>(P, sg.j0);
    sg.wid1 = unit_window<FMT>(P, sg.j1 - 1);
    sg.dst = 0;
    S.seg[f][lane] = sg;
  }
  if (lane == 0) S.nseg[f] = nseg;
}

// Cost prefix over the expert slots (one warp).
__device__ void cost_prefix(Shared &S, const FcPlan &P, int f) {
  const int lane = (int)lane_id();
  const int per = (S.na + 31) / 32;
  int sum = 0;
  for (int q = 0; q < per; ++q) {
    const int a = lane * per + q;
    if (a < S.na) sum += P.ct * pair_cost(P, S.slot[a].z);
  }
  int incl = sum;
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    const int v = __shfl_up_sync(0xFFFFFFFFu, incl, m);
    if (lane >= m) incl += v;
  }
  int run = incl - sum;
  for (int q = 0; q < per; ++q) {
    const int a = lane * per + q;
    if (a < S.na) {
      S.scum[f][a] = run;
      run += P.ct * pair_cost(P, S.slot[a].z);
    }
  }
  if (lane == 31) S.scum[f][S.na] = run;
}
// busy[f][c] = CTAs among [0, c) whose range is not empty (one warp).
__device__ void busy_prefix(Shared &S, int f) {
  const int lane = (int)lane_id(), G = (int)gridDim.x;
  const int per = (G + 31) / 32;
  int sum = 0;
  for (int q = 0; q < per; ++q) {
    const int c = lane * per + q;
    if (c < G) sum += S.bnd[f][c] < S.bnd[f][c + 1];
  }
  int incl = sum;
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    const int v = __shfl_up_sync(0xFFFFFFFFu, incl, m);
    if (lane >= m) incl += v;
  }
  int run = incl - sum;
  for (int q = 0; q < per; ++q) {
    const int c = lane * per + q;
    if (c < G) {
      S.busy[f][c] = (short)run;
      run += S.bnd[f][c] < S.bnd[f][c + 1];
    }
  }
  if (lane == 31) S.busy[f][G] = (short)run;
}

__device__ void split_bound(Shared &S, const FcPlan &P, int f, int c) {
  const int G = (int)gridDim.x, na = S.na;
  const int U = na * P.ct * P.ku;
  if (c >= G) {
    S.bnd[f][G] = U;
    return;
  }
  const int total = S.scum[f][na];
  const long long x = total < 0x7FFFFFFF / G ? (long long)((c * total) / G) : (long long)c * total / G;
  int lo = 0, hi = na - 1;  // the last slot whose prefix is <= x
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (S.scum[f][mid] <= x) lo = mid; else hi = mid - 1;
  }
  // inside slot lo: pairs of cost pc, each a pass-start charge then ku units
  // of cost cu; the range starts at the first unit that begins at or after x
  const int r = S.slot[lo].z, cu = unit_cost(P, r), pc = pair_cost(P, r);
  const long long rem = x - S.scum[f][lo];
  const int q = (int)(rem / pc);
  int u;
  if (q >= P.ct) {
    u = P.ct * P.ku;
  } else {
    const long long v = rem - (long long)q * pc - (long long)r * P.pass_cost;
    u = q * P.ku + (v <= 0 ? 0 : (int)min((long long)P.ku, (v + cu - 1) / cu));
  }
  S.bnd[f][c] = lo * P.ct * P.ku + u;
}

// Exclusive prefix of the partial-sum sizes of all (slot, tile) pairs of FC f (one warp).
__device__ void partial_bases(Shared &S, const FcPlan &P, int f) {
  const int lane = (int)lane_id();
  const int np = S.na * P.ct;
  const int per = (np + 31) / 32;
  int sum = 0;
  for (int q = 0; q < per; ++q) {
    const int p = lane * per + q;
    if (p < np) {
      const int cnt = busy_ctas(S, f, first_cta(S, P, f, p), last_cta(S, P, f, p) + 1);
      S.pcnt[f][p] = (short)cnt;
      sum += cnt * S.slot[p / P.ct].z * P.NT;
    }
  }
  int incl = sum;
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    const int v = __shfl_up_sync(0xFFFFFFFFu, incl, m);
    if (lane >= m) incl += v;
  }
  int run = incl - sum;
  for (int q = 0; q < per; ++q) {
    const int p = lane * per + q;
    if (p < np) {
      S.base[f][p] = run;
      run += S.pcnt[f][p] * S.slot[p / P.ct].z * P.NT;
    }
  }
  if (lane == 31) S.base[f][np] = run;
}

// ---- the copy warp --------------------------------------------------------------------

// Every unit of the CTA, FC1 then FC2, in consumption order; before the first
// unit of each scale window, that window's block scales (tensor copy).
// The two copy warps walk the same sequence of passes and units.  ROLE 0
// copies the weight units into the ring; ROLE 1 copies the FC1 activation
// rows and the scale windows, each blocking only on its own two slots, so
// that these small copies are issued a whole window ahead of their use
// instead of queueing behind the weight stream.
template <int FMT, int ROLE>
__device__ __noinline__ void producer(Shared &S, const LayerArgs &g, const LayerPlan &L, unsigned char *ring,
                                      uint8_t *stage, unsigned char *xraw) {
  constexpr int BS = FMT == QMOE_NVFP4 ? kNvfp4Block : kMxfp4Block;
  const int lane = (int)lane_id();
  const uint64_t pol = l2_evict_first_policy();
  // a wait by lane 0, its outcome in every lane: false once a bounded wait gave
  // up, after which this warp issues no further copy
  auto wait_all_lanes = [&](uint64_t *bar, uint32_t parity) -> bool {
    int ok = 1;
    if (lane == 0) ok = wait_bar(S, g, bar, parity) ? 1 : 0;
    return __shfl_sync(0xFFFFFFFFu, ok, 0) != 0;
  };
  // issue index of the last copy into each ring slot / window slot (drained before exit)
  uint32_t last_it[kRingMax] = {~0u, ~0u, ~0u, ~0u}, last_wn[2] = {~0u, ~0u};
  // With [E, N, K/bs] scales the weight stream starts once the first scale
  // window (a tensor copy, in the same bulk-copy queue) is on its way: small
  // copies issued behind a GPU-wide burst of bulk copies wait for all of it.
  // With k-major scales every small copy goes through cp.async and the
  // weight stream starts at once.
  bool first_done = ROLE == 0;
  // ROLE 1, once its first copies are issued: the global scales (needed after
  // the first grid barrier) and the partial-sum offsets (needed at the end of
  // the first pass), both off the consumers' path
  auto after_first = [&]() {
    if (lane == 0) mbar_arrive(&S.smallfirst);
    for (int i = lane; i < S.na; i += 32) {
      S.gs[0][i] = g.g1 ? __ldg(g.g1 + S.slot[i].x) : 1.0f;
      S.gs[1][i] = g.g2 ? __ldg(g.g2 + S.slot[i].x) : 1.0f;
    }
    mbar_arrive(&S.gsready);
    partial_bases(S, L.f[0], 0);
    partial_bases(S, L.f[1], 1);
    __syncwarp();
    // this CTA's partial-row offset in each of its segments
    for (int i = lane; i < S.nseg[0] + S.nseg[1]; i += 32) {
      const int f = i < S.nseg[0] ? 0 : 1, si = f == 0 ? i : i - S.nseg[0];
      const FcPlan &P = L.f[f];
      Seg &sg = S.seg[f][si];
      sg.dst = S.base[f][sg.pair] +
               busy_ctas(S, f, first_cta(S, P, f, sg.pair), (int)blockIdx.x) * S.slot[sg.a].z * P.NT;
    }
    mbar_arrive(&S.basesready);
    first_done = true;
  };
  uint32_t it = 0, wn = 0, xn = 0;
  if (ROLE == 0 && !L.f[0].kn) {
    if (!wait_all_lanes(&S.smallfirst, 0u)) goto drain;
  }
  for (int f = 0; f < 2; ++f) {
    const FcPlan &P = L.f[f];
    const uint8_t *wbase = f == 0 ? g.w1 : g.w2;
    const CUtensorMap *map = f == 0 ? &g.tm_s1 : &g.tm_s2;
    const uint32_t row_bytes = (uint32_t)(P.NT / 2);
    for (int si = 0; si < S.nseg[f]; ++si) {
      const Seg sg = S.seg[f][si];
      const int4 sd = S.slot[sg.a];
      const uint8_t *wexp = wbase + (size_t)sd.x * P.K * (P.N / 2) + (size_t)sg.t * row_bytes;
      const int col0 = sd.x * P.N + sg.t * P.NT;  // first scale row of the tile
      const int unit_k = 16 * P.RGS, xw_units = kXsK / unit_k;
      for (int c0 = 0; c0 < sd.z; c0 += kRowsMax) {
        const int rows_p = min(kRowsMax, sd.z - c0);
        int cur = -1;
        for (int j = sg.j0; j < sg.j1; ++j, ++it) {
          if (ROLE == 1 && f == 0 && (j - sg.j0) % xw_units == 0) {
            // FC1: the activation rows of this k window, ahead of its weights
            const int k0 = j * unit_k, len = min(P.K, min(sg.j1, j + xw_units) * unit_k) - k0;
            const int s = (int)(xn & 1u);
            if (xn >= 2u && !wait_all_lanes(&S.xempty[s], ((xn >> 1) + 1u) & 1u)) goto drain;
            // 16-byte pieces, all 32 lanes; each lane arrives once its own have landed
            const int cpr = len / 8;  // pieces per row
            for (int i = lane; i < rows_p * cpr; i += 32) {
              const int r = i / cpr, c = i - r * cpr;
              const int tok = S.row_tok[sd.y + c0 + r];
              cp_async16(xraw + (size_t)s * kXrawSlot + (size_t)r * kXsK * 2 + (size_t)c * 16,
                         g.x + (size_t)tok * g.H + k0 + (size_t)c * 8);
            }
            cp_async_arrive(&S.xfull[s]);
            ++xn;
          }
          const int wid = unit_window<FMT>(P, j);
          if (ROLE == 1 && P.tma && wid != cur) {
            const int s = (int)(wn & 1u);
            if (wn >= 2u && !wait_all_lanes(&S.wempty[s], ((wn >> 1) + 1u) & 1u)) goto drain;
            last_wn[s] = wn;
            uint8_t *dst = stage + (size_t)s * L.win_bytes;
            // the barrier counts 32 arrivals (one per lane, as for the cp.async windows)
            if (lane == 0) mbar_expect_tx(&S.wfull[s], (uint32_t)(P.NT * kTmaWB));
            else mbar_arrive(&S.wfull[s]);
            __syncwarp();
            for (int r = lane * P.box_rows; r < P.NT; r += 32 * P.box_rows)
              tensor_g2s_2d(dst + (size_t)r * kTmaWB, map, wid * kTmaWB, col0 + r, &S.wfull[s]);
            ++wn;
            cur = wid;
          }
          if (ROLE == 1) {
            if (!first_done) after_first();
            continue;
          }
          const uint32_t ring_n = (uint32_t)L.ring;
          const int s = (int)(it % ring_n);
          if (it >= ring_n && !wait_all_lanes(&S.empty[s], ((it / ring_n) + 1u) & 1u)) goto drain;
          last_it[s] = it;
          unsigned char *dst = ring + (size_t)s * L.slot_bytes;
          const int r0 = j * 16 * P.RGS, rows = unit_rows(P, j);
          // the slot was only read by the consumers (generic loads) before they
          // released it: no proxy fence is needed before the async copy writes it.
          // k-major scales: the unit's block rows travel in the same slot, at
          // bytes [sc_off, sc_off + nbu * NT), counted on the same barrier
          const int b0 = (r0 / BS), nbu = P.kn ? min(P.bpu, P.nblocks - b0) : 0;
          if (lane == 0) mbar_expect_tx(&S.full[s], (uint32_t)rows * row_bytes + (uint32_t)(nbu * P.NT));
          __syncwarp();
          if (P.kn) {
            const uint8_t *ssrc =
                (f == 0 ? g.s1 : g.s2) + ((size_t)sd.x * P.nblocks + b0) * P.N + (size_t)sg.t * P.NT;
            if (P.ct == 1) {
              if (lane == 31) bulk_g2s_stream(dst + P.sc_off, ssrc, (uint32_t)(nbu * P.NT), &S.full[s], pol);
            } else {
              for (int b = lane; b < nbu; b += 32)
                bulk_g2s_stream(dst + P.sc_off + (size_t)b * P.NT, ssrc + (size_t)b * P.N, (uint32_t)P.NT,
                                &S.full[s], pol);
            }
          }
          // row group rg (16 k rows) at dst + rg * rg_stride: the padding puts
          // the row groups read by one warp in different banks
          if (P.ct == 1) {
            const int nr = min(16, rows - 16 * lane);
            if (lane < P.RGS && nr > 0)
              bulk_g2s_stream(dst + (size_t)lane * P.rg_stride, wexp + (size_t)(r0 + 16 * lane) * row_bytes,
                              (uint32_t)nr * row_bytes, &S.full[s], pol);
          } else {
            for (int r = lane; r < rows; r += 32)
              bulk_g2s_stream(dst + (size_t)(r >> 4) * P.rg_stride + (size_t)(r & 15) * row_bytes,
                              wexp + (size_t)(r0 + r) * (P.N / 2), row_bytes, &S.full[s], pol);
          }
        }
      }
    }
  }
drain:
  if (!first_done) after_first();
  // No CTA may exit while its own copies are still landing in its shared
  // memory: wait (bounded, even after an abort) for the last copy issued into
  // every slot.  In a normal run the consumers have seen all of them already.
  if (ROLE == 1) asm volatile("cp.async.wait_all;" ::: "memory");
  if (lane == 0) {
    const uint32_t ring_n = (uint32_t)L.ring;
    for (int s = 0; s < (ROLE == 0 ? L.ring : 2); ++s) {
      const uint32_t last = ROLE == 0 ? last_it[s] : last_wn[s];
      if (last == ~0u) continue;
      uint64_t *bar = ROLE == 0 ? &S.full[s] : &S.wfull[s];
      const uint32_t parity = ROLE == 0 ? (last / ring_n) & 1u : (last >> 1) & 1u;
      uint32_t i = 0;
      while (!mbar_try_wait(bar, parity) && ++i < kWaitLimit) {
      }
    }
  }
  __syncwarp();
}

// ---- consumers -------------------------------------------------------------------------

// One k-group (16 rows x 8 columns) of a unit for one activation row: the 16
// words are loaded first, rows 4i, 4i+1 go to one set of 8 partial sums and
// rows 4i+2, 4i+3 to a second set (two independent FMA chains per column);
// the 16-row partial is multiplied once by its block scale.
template <int FMT, int RC>
__device__ __forceinline__ void consume_kg(const unsigned char *rows, int row_bytes, const __half *xb, uint2 sv,
                                           float (&acc)[RC][8]) {
  static_assert(RC == 1, "one row per pass");
  float sc[8];
  block_scales8<FMT>(sv, sc);
  uint32_t wv[16];
#pragma unroll
  for (int kk = 0; kk < 16; ++kk) wv[kk] = *reinterpret_cast<const uint32_t *>(rows + (size_t)kk * row_bytes);
  const uint4 xa = *reinterpret_cast<const uint4 *>(xb), xc = *reinterpret_cast<const uint4 *>(xb + 8);
  const uint32_t xx[8] = {xa.x, xa.y, xa.z, xa.w, xc.x, xc.y, xc.z, xc.w};
  float bp[8], bq[8];
#pragma unroll
  for (int c = 0; c < 8; ++c) bp[c] = bq[c] = 0.f;
#pragma unroll
  for (int kk = 0; kk < 16; kk += 4) {
    uint32_t p[4], q[4], r[4], t[4];
    dec8(wv[kk], p);
    dec8(wv[kk + 1], q);
    dec8(wv[kk + 2], r);
    dec8(wv[kk + 3], t);
    fma16(p, q, xx[kk >> 1], bp);
    fma16(r, t, xx[(kk >> 1) + 1], bq);
  }
#pragma unroll
  for (int c = 0; c < 8; ++c) acc[0][c] = fmaf(bp[c] + bq[c], sc[c], acc[0][c]);
}

struct PassCtx {
  int f, si, a, t, pair, c0, rows, j0, j1;
  int4 sd;
};

// Scale windows whose runs are not 16-byte aligned (no tensor copy): all
// consumer threads read window `wid` of the tile with byte loads into
// win[b][col].  Out of line, arguments by value.
template <int FMT>
__device__ __noinline__ void fill_window_cta(const LayerArgs &g, const LayerPlan &L, int f, int e, int t, int wid,
                                             uint8_t *win) {
  const FcPlan &P = L.f[f];
  const int b0 = wid * P.WB, nb = min(P.WB, P.nblocks - b0);
  cons_sync();  // nobody reads the previous window any more
  const uint8_t *scol = (f == 0 ? g.s1 : g.s2) + ((size_t)e * P.N + (size_t)t * P.NT) * P.nblocks + b0;
  const int groups = P.NT / 4, bgroups = (nb + 3) / 4;
  for (int job = threadIdx.x; job < groups * bgroups; job += kCons) {
    const int c4 = job / bgroups, bq = (job - c4 * bgroups) * 4;
    uint32_t v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint8_t *src = scol + (size_t)(4 * c4 + i) * P.nblocks + bq;
      uint32_t x = 0;
      for (int q = 0; q < 4 && bq + q < nb; ++q) x |= (uint32_t)__ldg(src + q) << (8 * q);
      v[i] = x;
    }
    store_tile4x4(v[0], v[1], v[2], v[3], win + (size_t)bq * P.NT + 4 * c4, P.NT, min(4, nb - bq));
  }
  cons_sync();
}

// A warp's share of a tensor-copied scale window: its 8 * WPW columns (stored
// [col][16 blocks] in the staging slot) transposed into its private area
// wp[b][col] (row stride 8 * WPW bytes), 4x4 byte tiles, two per lane.
__device__ __forceinline__ void warp_transpose_window(const uint8_t *wstage, uint8_t *wp, int warp, int wpw) {
  const int lane = threadIdx.x & 31;
  const int cols = 8 * wpw, cgroups = cols / 4;  // 4-column groups of this warp
  const uint8_t *src = wstage + (size_t)warp * cols * 16;
  for (int t = lane; t < cgroups * 4; t += 32) {
    const int cg = t % cgroups, bg = t / cgroups;
    uint32_t v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = *reinterpret_cast<const uint32_t *>(src + (size_t)(4 * cg + i) * 16 + 4 * bg);
    store_tile4x4(v[0], v[1], v[2], v[3], wp + (size_t)(4 * bg) * cols + 4 * cg, cols, 4);
  }
  __syncwarp();
}

// FC1 output column col of this row (row `row` of slot a): its partial sums
// summed in segment order.
__device__ __forceinline__ float fc1_column(const Shared &S, const LayerArgs &g, const FcPlan &P1, int a, int nrows,
                                            int row, int col) {
  const int t1 = col / P1.NT, c1 = col - t1 * P1.NT;
  const int pair = a * P1.ct + t1;
  const int nc = S.pcnt[0][pair];
  const size_t stride = (size_t)nrows * P1.NT;
  const float *src = g.p1 + S.base[0][pair] + (size_t)row * P1.NT + c1;
  float h = 0.f;
  for (int c = 0; c < nc; c += 8) {  // up to 8 loads in flight
    float v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) v[u] = c + u < nc ? __ldcg(src + (c + u) * stride) : 0.f;
#pragma unroll
    for (int u = 0; u < 8; ++u)
      if (c + u < nc) h += v[u];
  }
  return h;
}

// a[row][k] = bf16(SwiGLU(g1 * h)) for FC2's activations, h = the FC1 partial
// sums of this row (row c0 + rr of slot a) summed in segment order.  The gate
// and linear columns are 2k and 2k + 1 (interleaved, read as one pair), or k
// and I + k (concatenated).
__device__ __forceinline__ uint16_t fc2_activation(const Shared &S, const LayerArgs &g, const LayerPlan &L, int a,
                                                   int nrows, int row, int k) {
  const FcPlan &P1 = L.f[0];
  if (g.fusion == 2) {
    const float g1 = S.gs[0][a];
    const float hg = fc1_column(S, g, P1, a, nrows, row, k), hl = fc1_column(S, g, P1, a, nrows, row, g.I + k);
    return (uint16_t)f32_to_bf16_rne(swiglu(hg * g1, hl * g1, g.alpha, g.beta, g.limit));
  }
  const int col = 2 * k;
  const int t1 = col / P1.NT, c1 = col - t1 * P1.NT;
  const int pair = a * P1.ct + t1;
  const int nc = S.pcnt[0][pair];
  const size_t stride = (size_t)nrows * P1.NT;
  const float *src = g.p1 + S.base[0][pair] + (size_t)row * P1.NT + c1;
  float hg = 0.f, hl = 0.f;
  for (int c = 0; c < nc; c += 8) {  // up to 8 loads in flight, summed in segment order
    float2 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u)
      v[u] = c + u < nc ? __ldcg(reinterpret_cast<const float2 *>(src + (c + u) * stride)) : make_float2(0.f, 0.f);
#pragma unroll
    for (int u = 0; u < 8; ++u)
      if (c + u < nc) { hg += v[u].x; hl += v[u].y; }
  }
  const float g1 = S.gs[0][a];
  return (uint16_t)f32_to_bf16_rne(swiglu(hg * g1, hl * g1, g.alpha, g.beta, g.limit));
}

// Activation rows [c0, c0 + rows) of the pass, k in [k0, k0 + len), as fp16
// with a per-row power-of-two rescale, into this warp's own window xw
// (row stride kXsK): every warp reads the raw bf16 rows and converts them
// itself, so no CTA barrier is needed.  Raw rows come from: FC1, raw slot
// xn & 1 (bulk-copied by the copy warp); FC2, the pre-staged buffer (row
// stride len) at pre_off, or, when pre-staging did not fit, they are first
// computed from the FC1 partials by all consumer threads into the raw buffer.
template <int RC>
__device__ __forceinline__ void stage_warp(Shared &S, const LayerArgs &g, const LayerPlan &L, const PassCtx &C,
                                           int k0, int len, __half *xw, unsigned char *xraw, uint32_t &xn,
                                           int &pre_off, int (&sh)[RC]) {
  const int lane = threadIdx.x & 31;
  const uint16_t *src;
  int stride = kXsK;
  if (C.f == 0) {
    const int s = (int)(xn & 1u);
    wait_bar(S, g, &S.xfull[s], (xn >> 1) & 1u);
    src = reinterpret_cast<const uint16_t *>(xraw + (size_t)s * kXrawSlot);
  } else if (S.fc2_pre) {
    src = reinterpret_cast<const uint16_t *>(xraw) + pre_off;
    stride = len;
    pre_off += C.rows * len;
  } else {
    cons_sync();  // every warp is done with the raw buffer
    uint16_t *xb = reinterpret_cast<uint16_t *>(xraw);
    for (int i = threadIdx.x; i < C.rows * len; i += kCons) {
      const int rr = i / len, kk = i - rr * len;
      xb[(size_t)rr * kXsK + kk] = fc2_activation(S, g, L, C.a, C.sd.z, C.c0 + rr, k0 + kk);
    }
    cons_sync();
    src = xb;
  }
  __syncwarp();  // this warp is done with its previous window
#pragma unroll
  for (int r = 0; r < RC; ++r) {
    uint32_t m = 0;
    if (r < C.rows)
      for (int q = lane; q * 8 < len; q += 32)
        m = max(m, absmax_bf16x8(*reinterpret_cast<const uint4 *>(src + (size_t)r * stride + 8 * q)));
    m = __reduce_max_sync(0xFFFFFFFFu, m);
    sh[r] = row_shift(m);
    const float f = pow2f(-sh[r]);
    for (int q = lane; q * 8 < len; q += 32) {
      const uint4 v = r < C.rows ? *reinterpret_cast<const uint4 *>(src + (size_t)r * stride + 8 * q)
                                 : make_uint4(0, 0, 0, 0);
      reinterpret_cast<uint4 *>(xw + (size_t)r * kXsK)[q] = bf16x8_to_f16x8(v, f);
    }
  }
  __syncwarp();
  if (C.f == 0) {
    if (lane == 0) mbar_arrive(&S.xempty[xn & 1u]);
    ++xn;
  }
}

// FC2's activations of every pass of this CTA, computed once right after the
// first grid barrier (while the memory system is quiet) into the raw buffer,
// pass after pass, row stride = the pass's k length.  Returns false (nothing
// staged) when a pass needs more than one staging window or the buffer is
// too small.
__device__ bool prestage_fc2(Shared &S, const LayerArgs &g, const LayerPlan &L, unsigned char *xraw) {
  const FcPlan &P = L.f[1];
  const int unit_k = 16 * P.RGS;
  int total = 0;
  for (int si = 0; si < S.nseg[1]; ++si) {
    const Seg sg = S.seg[1][si];
    const int len = min(P.K, sg.j1 * unit_k) - sg.j0 * unit_k;
    if (len > kXsK) return false;
    total += S.slot[sg.a].z * len;
  }
  if (total * 2 > kXrawBytes) return false;
  // one flat loop over every element of every pass, so that all their
  // partial-sum loads are in flight together (segment after segment, a
  // segment's rows after one another: the passes' order)
  uint16_t *dst = reinterpret_cast<uint16_t *>(xraw);
  for (int i = threadIdx.x; i < total; i += kCons) {
    int base = 0;
    for (int si = 0; si < S.nseg[1]; ++si) {
      const Seg sg = S.seg[1][si];
      const int rows = S.slot[sg.a].z;
      const int k0 = sg.j0 * unit_k, len = min(P.K, sg.j1 * unit_k) - k0;
      if (i < base + rows * len) {
        const int rr = (i - base) / len, kk = i - base - rr * len;
        dst[i] = fc2_activation(S, g, L, sg.a, rows, rr, k0 + kk);
        break;
      }
      base += rows * len;
    }
  }
  return true;
}

// One pass (rows [c0, c0 + rows) of a segment).  Thread mapping: a warp owns
// WPW = 32 / RGS column words (8 columns each) over all RGS row groups,
// lane = rg * WPW + wl; the row-group partial sums are combined with warp
// shuffles, so the pass needs no CTA barrier.
template <int FMT, int RC, int KN>
__device__ __forceinline__ void run_pass(Shared &S, const LayerArgs &g, const LayerPlan &L, const PassCtx &C,
                                         unsigned char *ring, uint8_t *win, const uint8_t *stage, __half *xw,
                                         unsigned char *xraw, uint32_t &it, uint32_t &wn, uint32_t &xn,
                                         int &pre_off, uint32_t &slot, uint32_t &phase) {
  const FcPlan &P = L.f[C.f];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // RGS is a power of two: the lane geometry by shifts, no division
  const int lg_rgs = __ffs(P.RGS) - 1, wpw = 32 >> lg_rgs, lg_wpw = 5 - lg_rgs;
  const int rg = lane >> lg_wpw, wl = lane & (wpw - 1);
  const int w = warp * wpw + wl;
  const bool active = w < P.NW;
  const int row_bytes = P.NT / 2;
  constexpr int BS = FMT == QMOE_NVFP4 ? kNvfp4Block : kMxfp4Block;
  float acc[RC][8];
#pragma unroll
  for (int r = 0; r < RC; ++r)
#pragma unroll
    for (int c = 0; c < 8; ++c) acc[r][c] = 0.f;
  int sh[RC];
#pragma unroll
  for (int r = 0; r < RC; ++r) sh[r] = 0;
  const int unit_k = 16 * P.RGS;
  const int xw_units = kXsK / 16 >> lg_rgs;  // kXsK / unit_k
  int cur_wid = -1;
  uint32_t ws = 0;
  // ring position (slot, phase) of the pass's first unit: carried from pass
  // to pass by the caller and advanced without division
  const uint32_t ring_n = (uint32_t)L.ring;
  // k-major scales: this lane's 8 scale bytes sit at a fixed offset in every slot
  const int sc_lane = P.sc_off + ((rg * 16) / BS) * P.NT + 8 * w;
  for (int xj = C.j0; xj < C.j1; xj += xw_units) {
    const int xj1 = min(C.j1, xj + xw_units);
    const int k0 = xj * unit_k, len = min(P.K, xj1 * unit_k) - k0;
    int nsh[RC];
    stage_warp<RC>(S, g, L, C, k0, len, xw, xraw, xn, pre_off, nsh);
    if (xj != C.j0) {
#pragma unroll
      for (int r = 0; r < RC; ++r)
#pragma unroll
        for (int c = 0; c < 8; ++c) acc[r][c] = ldexp2(acc[r][c], sh[r] - nsh[r]);
    }
#pragma unroll
    for (int r = 0; r < RC; ++r) sh[r] = nsh[r];
    for (int j = xj; j < xj1; ++j, ++it) {
      if (KN) {  // k-major scales come with the unit: no windows
        wait_bar(S, g, &S.full[slot], phase);
        const int kg = j * P.RGS + rg;
        const unsigned char *sb = ring + (size_t)slot * L.slot_bytes;
        if (active && kg < P.nkg)
          consume_kg<FMT, RC>(sb + (size_t)rg * P.rg_stride + 4 * w, row_bytes, xw + (kg * 16 - k0),
                              *reinterpret_cast<const uint2 *>(sb + sc_lane), acc);
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.empty[slot]);
        if (++slot == ring_n) {
          slot = 0;
          phase ^= 1u;
        }
        continue;
      }
      const int wid = unit_window<FMT>(P, j);
      if (wid != cur_wid) {
        if (P.tma) {
          ws = wn & 1u;
          wait_bar(S, g, &S.wfull[ws], (wn >> 1) & 1u);
          __syncwarp();  // the warp's previous window is no longer read
          // warps that own columns (NW is a multiple of WPW for tensor-copied
          // windows, so these private areas fill exactly 16 * NT bytes)
          if (warp * wpw < P.NW)
            warp_transpose_window(stage + (size_t)ws * L.win_bytes, win + (size_t)warp * kTmaWB * 8 * wpw, warp, wpw);
          // the staging slot can go back at once: this warp has its own copy
          if (lane == 0) mbar_arrive(&S.wempty[ws]);
          ++wn;
        } else {
          fill_window_cta<FMT>(g, L, C.f, C.sd.x, C.t, wid, win);
        }
        cur_wid = wid;
      }
      const int s = (int)(it % (uint32_t)L.ring);
      wait_bar(S, g, &S.full[s], (it / (uint32_t)L.ring) & 1u);
      const int kg = j * P.RGS + rg;
      if (active && kg < P.nkg) {
        const unsigned char *rows = ring + (size_t)s * L.slot_bytes + (size_t)rg * P.rg_stride + 4 * w;
        const int blk = (kg * 16) / BS - cur_wid * P.WB;
        const uint2 sv = P.tma ? *reinterpret_cast<const uint2 *>(win + (size_t)warp * kTmaWB * 8 * wpw +
                                                                   (size_t)blk * 8 * wpw + 8 * wl)
                               : *reinterpret_cast<const uint2 *>(win + (size_t)blk * P.NT + 8 * w);
        consume_kg<FMT, RC>(rows, row_bytes, xw + (kg * 16 - k0), sv, acc);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.empty[s]);
    }
  }
  // combine the row groups (a fixed butterfly over the lanes of the warp) and
  // write the partial rows
  for (int m = wpw; m < 32; m <<= 1)
#pragma unroll
    for (int r = 0; r < RC; ++r)
#pragma unroll
      for (int c = 0; c < 8; ++c) acc[r][c] += __shfl_xor_sync(0xFFFFFFFFu, acc[r][c], m);
  // partial rows of this segment: dst[row * NT + col], row = c0 + r (the
  // offsets are computed by the activation copy warp after its first copies)
  wait_bar(S, g, &S.basesready, 0u);
  float *dst = (C.f == 0 ? g.p1 : g.p2) + S.seg[C.f][C.si].dst;
  if (active && rg == 0) {
#pragma unroll
    for (int r = 0; r < RC; ++r) {
      if (r < C.rows) {
        // the sum is near the rescaled row's magnitude (the block scales
        // enter at their own value), so undoing the 2^-shift cannot underflow
        const float un = pow2f(sh[r]);
        float4 *d = reinterpret_cast<float4 *>(dst + (size_t)(C.c0 + r) * P.NT + 8 * w);
        d[0] = make_float4(acc[r][0] * un, acc[r][1] * un, acc[r][2] * un, acc[r][3] * un);
        d[1] = make_float4(acc[r][4] * un, acc[r][5] * un, acc[r][6] * un, acc[r][7] * un);
      }
    }
  }
}

// out[t][n] = bf16(sum_j w[t][j] * g2 * y_j[n]), once every FC2 partial is
// written: 8 lanes per column pair, lane j gathers expert j's FC2 partials; the
// lanes are summed by a fixed butterfly.
__device__ __noinline__ void finalize(Shared &S, const LayerArgs &g, const LayerPlan &L) {
  const FcPlan &P2 = L.f[1];
  const int half = g.H / 2;
  const int items = g.T * half * 8;
  const int items_pad = (items + 31) & ~31;
  for (int idx = (int)blockIdx.x * kCons + (int)threadIdx.x; idx < items_pad; idx += (int)gridDim.x * kCons) {
    const int grp = idx >> 3, j = idx & 7;
    const bool ok = grp < g.T * half && j < g.k;
    float y0 = 0.f, y1 = 0.f;
    int t = 0, n = 0;
    if (ok) {
      t = grp / half;
      n = 2 * (grp - t * half);
      const int ex = t * g.k + j;
      const int p = S.r_e2p[ex];
      const int a = S.row2slot[p];
      const int4 sd = S.slot[a];
      const int t2 = n / P2.NT, col = n - t2 * P2.NT;
      const int pair = a * P2.ct + t2;
      const int nc = S.pcnt[1][pair];
      const size_t stride = (size_t)sd.z * P2.NT;
      const float *src = g.p2 + S.base[1][pair] + (size_t)(p - sd.y) * P2.NT + col;
      float s0 = 0.f, s1 = 0.f;
      for (int c = 0; c < nc; c += 8) {  // up to 8 loads in flight, summed in segment order
        float2 v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u)
          v[u] = c + u < nc ? __ldcg(reinterpret_cast<const float2 *>(src + (c + u) * stride)) : make_float2(0.f, 0.f);
#pragma unroll
        for (int u = 0; u < 8; ++u)
          if (c + u < nc) { s0 += v[u].x; s1 += v[u].y; }
      }
      const float wgt = S.r_w[ex], g2 = S.gs[1][a];
      y0 = wgt * (s0 * g2);
      y1 = wgt * (s1 * g2);
    }
#pragma unroll
    for (int m = 4; m > 0; m >>= 1) {
      y0 += __shfl_xor_sync(0xFFFFFFFFu, y0, m);
      y1 += __shfl_xor_sync(0xFFFFFFFFu, y1, m);
    }
    if (ok && j == 0)
      reinterpret_cast<uint32_t *>(g.out + (size_t)t * g.H)[n / 2] = f32_to_bf16_rne(y0) | (f32_to_bf16_rne(y1) << 16);
  }
}

template <int FMT, int KN>
__device__ __noinline__ void consumer(Shared &S, const LayerArgs &g, const LayerPlan &L, unsigned char *ring,
                                      uint8_t *win, const uint8_t *stage, __half *xs, unsigned char *xraw) {
  uint32_t it = 0, wn = 0, xn = 0;
  uint32_t slot = 0, phase = 0;  // ring position of unit `it` (k-major path)
  __half *xw = xs + (size_t)(threadIdx.x >> 5) * (kXwBytes / 2);  // this warp's activation window
  int pre_off = 0;
  for (int f = 0; f < 2; ++f) {
    if (f == 1) {
      grid_barrier(S, g, g.meta + 2);  // every FC1 partial is written
      wait_bar(S, g, &S.gsready, 0u);
      const bool pre = prestage_fc2(S, g, L, xraw);
      if (threadIdx.x == 0) S.fc2_pre = pre ? 1 : 0;
      cons_sync();
    }
    for (int si = 0; si < S.nseg[f]; ++si) {
      const Seg sg = S.seg[f][si];
      PassCtx C;
      C.f = f;
      C.si = si;
      C.pair = sg.pair;
      C.a = sg.a;
      C.t = sg.t;
      C.sd = S.slot[sg.a];
      C.j0 = sg.j0;
      C.j1 = sg.j1;
      for (int c0 = 0; c0 < C.sd.z; c0 += kRowsMax) {
        C.c0 = c0;
        C.rows = min(kRowsMax, C.sd.z - c0);
        run_pass<FMT, kRowsMax, KN>(S, g, L, C, ring, win, stage, xw, xraw, it, wn, xn, pre_off, slot, phase);
      }
    }
  }
  grid_barrier(S, g, g.meta + 3);  // every FC2 partial is written
  if (threadIdx.x == 0) leave_counters(g);
  finalize(S, g, L);
}

template <int FMT>
__global__ void __launch_bounds__(kLayerThreads, 1) moe_layer_kernel(const __grid_constant__ LayerArgs g,
                                                                   const __grid_constant__ LayerPlan L) {
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ Shared S;
  const int tid = threadIdx.x, warp = tid >> 5;
  // Launched with programmatic dependent launch, the kernel may start while
  // the previous kernel of the stream still runs: nothing in global memory
  // (inputs, workspace) is touched before that kernel's results are visible.
  // The next kernel may then be scheduled at once: it is launched only once
  // every CTA of this grid has passed this point (so all are resident), and
  // it cannot become resident on an SM before this kernel's CTA there exits.
  pdl_wait();
  pdl_launch_dependents();
  if (tid == 0) {
    for (int i = 0; i < kRingMax; ++i) {
      mbar_init(&S.full[i], 1);
      mbar_init(&S.empty[i], kConsWarps);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&S.wfull[i], 32);  // one arrival per lane of the activation/scale-copy warp
      mbar_init(&S.wempty[i], kConsWarps);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&S.xfull[i], 32);
      mbar_init(&S.xempty[i], kConsWarps);
    }
    mbar_init(&S.gsready, 32);
    mbar_init(&S.smallfirst, 1);
    mbar_init(&S.basesready, 32);
    mbar_fence_init();
    S.abort = 0;
    S.fc2_pre = 0;
  }
  // Routing, in every CTA with the routing kernel's top-k code (so every CTA
  // holds the same, bit-identical result and no separate launch is needed):
  // warp w routes tokens w, w + 18, ...; then one warp ranks the T * k <= 64
  // rows by expert into the maps and the active-expert slots and forms the
  // cost prefix of both FCs over those slots.
  const int R = g.T * g.k;
  for (int t = warp; t < g.T; t += kLayerThreads / 32) {
    if (g.route_n == 1) route_one_token<1>(g.logits, g.mix, t, g.E, g.k, g.normalize, S.r_ids, S.r_w);
    else if (g.route_n == 2) route_one_token<2>(g.logits, g.mix, t, g.E, g.k, g.normalize, S.r_ids, S.r_w);
    else if (g.route_n == 4) route_one_token<4>(g.logits, g.mix, t, g.E, g.k, g.normalize, S.r_ids, S.r_w);
    else route_one_token<8>(g.logits, g.mix, t, g.E, g.k, g.normalize, S.r_ids, S.r_w);
  }
  __syncthreads();
  if (warp == 0) {
    RankOut o;
    o.e2p = S.r_e2p;
    o.p2e = S.r_p2e;
    o.row_tok = S.row_tok;
    o.row2slot = S.row2slot;
    o.slots = S.slot;
    o.na = &S.na;
    rank_rows_small(S.r_ids, R, g.E, g.k, o);
    __syncwarp();
    if (S.na > 0) {
      cost_prefix(S, L.f[0], 0);
      cost_prefix(S, L.f[1], 1);
    }
  } else if (blockIdx.x == 0 && g.ids_out && tid - 32 < R) {
    g.ids_out[tid - 32] = S.r_ids[tid - 32];
  }
  __syncthreads();
  const int na = min(S.na, kMaxSlots);
  if (na <= 0) return;  // every CTA sees the same count
  {  // the split of both FCs, one boundary per thread
    const int G = (int)gridDim.x;
    if (tid <= G) split_bound(S, L.f[0], 0, tid);
    else if (tid <= 2 * G + 1) split_bound(S, L.f[1], 1, tid - G - 1);
  }
  __syncthreads();
  // this CTA's segments, and (beside them) the CTAs holding units, which the
  // partial-sum offsets need
  if (warp == 0) build_segments<FMT>(S, g, L.f[0], 0);
  else if (warp == 1) build_segments<FMT>(S, g, L.f[1], 1);
  else if (warp == 2 || warp == 3) busy_prefix(S, warp - 2);
  __syncthreads();
  // 1 KB-aligned regions (the tensor and bulk copies need 16-byte alignment)
  unsigned char *base = smem + ((1024u - (smem_addr(smem) & 1023u)) & 1023u);
  unsigned char *ring = base;
  uint8_t *win = base + L.sw_off;
  uint8_t *stage = base + L.st_off;
  __half *xs = reinterpret_cast<__half *>(base + L.xs_off);
  unsigned char *xraw = base + L.xr_off;
  if (warp == kWarpW)
    producer<FMT, 0>(S, g, L, ring, stage, xraw);
  else if (warp == kWarpS)
    producer<FMT, 1>(S, g, L, ring, stage, xraw);
  else if (L.f[0].kn)  // both FCs share the scale layout
    consumer<FMT, 1>(S, g, L, ring, win, stage, xs, xraw);
  else
    consumer<FMT, 0>(S, g, L, ring, win, stage, xs, xraw);
}

// ---- host side ---------------------------------------------------------------------------

static bool make_fc_plan(int fmt, bool kn, int K, int N, int BS, FcPlan &P) {
  const int nblocks = K / BS;
  // tensor-copied scale windows ([E, N, nblocks] scales): NVFP4 (one block
  // per k-group, so a thread needs 16 / RGS <= 4 blocks of a window) with
  // whole 16-block windows.  k-major scales need no tensor copy.
  bool tma = !kn && fmt == QMOE_NVFP4 && nblocks % kTmaWB == 0;
  int best_busy = 0;
  P = FcPlan{};
  for (int ct = 1; ct <= kMaxTiles; ++ct) {
    if (N % ct) continue;
    const int NT = N / ct;
    if (NT % 32) continue;
    if (tma && (NT > kTmaMaxNT || NT % 64)) continue;
    const int NW = NT / 8;
    if (NW > kCons) continue;
    int RGS = 1;
    while (NW * RGS * 2 <= kCons && RGS < 16) RGS *= 2;
    if (NW * RGS > best_busy) {
      best_busy = NW * RGS;
      P.ct = ct;
      P.NT = NT;
      P.NW = NW;
      P.RGS = RGS;
    }
  }
  if (best_busy == 0) {
    if (!tma) return false;
    return make_fc_plan(QMOE_MXFP4 + 1, false, K, N, BS, P);  // no tensor-copy tiling: plain windows
  }
  P.K = K;
  P.N = N;
  P.nkg = K / 16;
  P.ku = (P.nkg + P.RGS - 1) / P.RGS;
  P.nblocks = nblocks;
  P.tma = tma ? 1 : 0;
  P.kn = kn ? 1 : 0;
  P.bpu = (P.RGS * 16) / BS > 0 ? (P.RGS * 16) / BS : 1;  // block rows a unit touches (k-major scales)
  int WB = kTmaWB;
  if (!tma)
    while (WB * P.NT > kMaxWinBytes) WB /= 2;
  const int bpu = (P.RGS * 16) / BS > 0 ? (P.RGS * 16) / BS : 1;
  if (WB < bpu) return false;
  P.WB = WB;
  P.box_rows = 256;
  while (P.NT % P.box_rows) P.box_rows /= 2;
  // row groups in a ring slot: 16 rows + a pad of 16 * max(1, WPW / 4) bytes,
  // so that the WPW words x RGS row groups one warp reads fall in different
  // banks (conflict-free for WPW >= 4)
  const int wpw = 32 / P.RGS > 0 ? 32 / P.RGS : 1;
  P.rg_stride = 16 * (P.NT / 2) + 16 * (wpw / 4 > 1 ? wpw / 4 : 1);
  P.sc_off = P.RGS * P.rg_stride;  // k-major scales after the unit's row groups (16-byte aligned)
  if (tma && (P.box_rows < 64 || P.RGS < 4 || P.NW % (32 / P.RGS) != 0)) {  // whole warps of columns
    return make_fc_plan(QMOE_MXFP4 + 1, false, K, N, BS, P);
  }
  return true;
}

qmoe_status make_layer_plan(int fmt, bool kmajor, int T, int H, int I, int E, int k, LayerPlan &L,
                            size_t &p1_floats, size_t &p2_floats) {
  const int BS = block_size(fmt);
  L = LayerPlan{};
  if (!make_fc_plan(fmt, kmajor, H, 2 * I, BS, L.f[0]) || !make_fc_plan(fmt, kmajor, I, H, BS, L.f[1])) {
    set_error("no column tiling of N = %d / %d fits the decode kernel", 2 * I, H);
    return QMOE_ERR_UNSUPPORTED;
  }
  const size_t G = (size_t)num_sms();
  if (G > (size_t)kMaxCtas) {
    set_error("the decode kernel supports at most %d SMs (this GPU has %zu)", kMaxCtas, G);
    return QMOE_ERR_UNSUPPORTED;
  }
  const size_t R = (size_t)T * k;
  const size_t na_max = std::min<size_t>((size_t)E, R);
  // pass-start charge of the split, in 1/64 of a unit decoded for one row
  // (fitted to per-CTA timings), and the per-unit cost of an r-row expert:
  // with n1 = R * ct * ku / G one-row units per CTA (in [1, ku]) and
  // p = pass_cost / 64, a CTA inside an r-row pair matches a one-row CTA's
  // time (n1 + p) with n_r = (n1 - p * (r - 1)) / r units, so a unit costs
  // 64 * n1 / n_r, at most twice the decode alone (a pair of many rows is
  // then cut into short segments, each still paying all its rows' passes)
  const int pass_start[2] = {192, 96};
  for (int f = 0; f < 2; ++f) {
    FcPlan &P = L.f[f];
    P.pass_cost = pass_start[f];
    const double n1 = std::max(1.0, std::min((double)P.ku, (double)(R * P.ct * P.ku) / (double)G));
    const double p = P.pass_cost / 64.0;
    for (int r = 1; r <= kCostRows; ++r) {
      const double nr = (n1 - p * (r - 1)) / r;
      const double c = nr > n1 / (2.0 * r) ? 64.0 * n1 / nr : 128.0 * r;
      P.ucost[r - 1] = (int)std::min(128.0 * r, std::ceil(c));
    }
  }
  int slot = 0, win = 0;
  for (int f = 0; f < 2; ++f) {
    const FcPlan &P = L.f[f];
    slot = std::max(slot, P.RGS * P.rg_stride + (P.kn ? P.bpu * P.NT : 0));
    win = std::max(win, (P.tma ? kTmaWB : P.WB) * P.NT);
    // segments of one CTA: at most the pairs that exist, and at most two more
    // (the first and the last) than the pairs lying wholly inside its cost
    // range [c * total / G, (c + 1) * total / G], each of which costs at
    // least pass_cost + 64 ku (one row).  A unit of an r-row expert costs at
    // most 128 r, so the total is at most ct * R * (pass_cost + 128 ku).
    const size_t pc_min = (size_t)P.pass_cost + 64 * (size_t)P.ku;
    const size_t total = (size_t)P.ct * R * ((size_t)P.pass_cost + 128 * (size_t)P.ku);
    const size_t segs = std::min<size_t>(na_max * (size_t)P.ct, 2 + (total / G + 1) / pc_min);
    if (segs > (size_t)kMaxSegs) {
      set_error("too many experts per CTA for the decode kernel (N = %d, K = %d)", P.N, P.K);
      return QMOE_ERR_UNSUPPORTED;
    }
  }
  L.slot_bytes = (slot + 1023) & ~1023;
  L.win_bytes = (win + 1023) & ~1023;
  // the consumers' own window area: not needed when both FCs read k-major
  // windows in place from the staging slots
  const bool kn = L.f[0].kn && L.f[1].kn;  // no window buffers: scales ride in the ring
  if (kn) L.win_bytes = 0;
  const bool own_win = !kn;
  // the deepest weight ring that fits next to everything else (a deeper ring
  // keeps more bytes in flight per SM)
  const int limit = kSmemOptin - (int)sizeof(Shared) - 1024;
  for (L.ring = kRingMax; L.ring >= 3; --L.ring) {
    L.sw_off = L.ring * L.slot_bytes;
    L.st_off = L.sw_off + (own_win ? L.win_bytes : 0);
    L.xs_off = L.st_off + 2 * L.win_bytes;
    L.xr_off = L.xs_off + kConsWarps * kXwBytes;
    L.smem = L.xr_off + kXrawBytes + 1024;  // + room to align the base to 1 KB
    if (L.smem <= limit) break;
  }
  if (L.ring < 3) {
    set_error("the decode kernel's buffers do not fit in shared memory (N = %d / %d)", 2 * I, H);
    return QMOE_ERR_UNSUPPORTED;
  }
  // Partial rows: every (slot, tile) pair once, plus one more segment of at
  // most T rows at each boundary between two CTAs.
  const size_t rows_max = std::min<size_t>((size_t)T, R);
  p1_floats = (R * L.f[0].ct + (G - 1) * rows_max) * L.f[0].NT;
  p2_floats = (R * L.f[1].ct + (G - 1) * rows_max) * L.f[1].NT;
  return QMOE_OK;
}

// Tensor map of one FC's block scales viewed as a 2-D byte array: E*N rows of
// nblocks bytes; box = 16 blocks x box_rows rows, stored densely (the 16-byte
// row of column c at byte 16 c of the window).
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static cudaError_t encode_scale_map(CUtensorMap *m, const uint8_t *scales, int E, const FcPlan &P) {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q);
    if (err != cudaSuccess || q != cudaDriverEntryPointSuccess || !p) {
      set_error("cuTensorMapEncodeTiled is not available");
      return err != cudaSuccess ? err : cudaErrorNotSupported;
    }
    fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  const cuuint64_t dims[2] = {(cuuint64_t)P.nblocks, (cuuint64_t)E * (cuuint64_t)P.N};
  const cuuint64_t strides[1] = {(cuuint64_t)P.nblocks};
  const cuuint32_t box[2] = {(cuuint32_t)kTmaWB, (cuuint32_t)P.box_rows};
  const cuuint32_t es[2] = {1, 1};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(scales), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_error("cuTensorMapEncodeTiled failed (%d)", (int)r);
    return cudaErrorInvalidValue;
  }
  return cudaSuccess;
}

template <int FMT>
static cudaError_t launch_layer_fmt(const LayerArgs &a, const LayerPlan &L, bool pdl, cudaStream_t stream) {
  // kernel attributes are per device: the opt-in size set and the size checked for residency
  static std::atomic<int> smem_set[kMaxDevices], smem_ok[kMaxDevices];
  const int dev = current_device();
  if (dev < 0) return cudaErrorInvalidDevice;
  auto kfn = moe_layer_kernel<FMT>;
  if (L.smem > smem_set[dev].load(std::memory_order_acquire)) {
    cudaError_t err = cudaFuncSetAttribute(kfn, cudaFuncAttributePreferredSharedMemoryCarveout,
                                           cudaSharedmemCarveoutMaxShared);
    if (err != cudaSuccess) return err;
    err = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, L.smem);
    if (err != cudaSuccess) return err;
    smem_set[dev].store(L.smem, std::memory_order_release);
  }
  if (L.smem != smem_ok[dev].load(std::memory_order_acquire)) {  // one CTA per SM must fit, or the cooperative launch is refused
    int per_sm = 0;
    cudaError_t err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kfn, kLayerThreads, L.smem);
    if (err != cudaSuccess) return err;
    if (per_sm < 1) {
      cudaFuncAttributes fa{};
      cudaFuncGetAttributes(&fa, kfn);
      set_error("decode kernel does not fit on an SM: %d registers x %d threads, %zu + %d bytes shared memory",
                fa.numRegs, kLayerThreads, (size_t)fa.sharedSizeBytes, L.smem);
      return cudaErrorCooperativeLaunchTooLarge;
    }
    smem_ok[dev].store(L.smem, std::memory_order_release);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_sms());
  cfg.blockDim = dim3(kLayerThreads);
  cfg.dynamicSmemBytes = L.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kfn, a, L);
}

cudaError_t launch_layer(LayerArgs &a, const LayerPlan &L, int E, bool pdl, cudaStream_t stream) {
  if (L.f[0].tma) {
    cudaError_t err = encode_scale_map(&a.tm_s1, a.s1, E, L.f[0]);
    if (err != cudaSuccess) return err;
  }
  if (L.f[1].tma) {
    cudaError_t err = encode_scale_map(&a.tm_s2, a.s2, E, L.f[1]);
    if (err != cudaSuccess) return err;
  }
  if (a.fmt == QMOE_NVFP4) return launch_layer_fmt<QMOE_NVFP4>(a, L, pdl, stream);
  return launch_layer_fmt<QMOE_MXFP4>(a, L, pdl, stream);
}

}  // namespace qmoe

extern "C" int qmoe_binary_version(void) {
  cudaFuncAttributes fa{};
  if (cudaFuncGetAttributes(&fa, qmoe::moe_layer_kernel<QMOE_NVFP4>) != cudaSuccess) return -1;
  return fa.binaryVersion;
}
