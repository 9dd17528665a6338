// Decode path of the FP4 MoE layer for k-major block scales ([E, K/bs, N]):
// top-k softmax routing and the permute maps, FC1 GEMV with SwiGLU, FC2 GEMV
// and the weighted un-permute in one persistent kernel, the E2M1 weights
// dequantised in registers.
//
// The method is the operator's ("MoE and QMoE - CUDA Operator Documentation"
// §1 routing / permute / finalize, §8 SwiGLU, §9b NVFP4); the GEMV design
// follows the decode-GEMV pull request ("[CUDA] Speed up the NVFP4 QMoE
// decode GEMV and enable it for MTP verify": coalesced weight and scale
// streams, loads batched ahead of their decode, table-free E2M1 decode,
// block scale applied to a per-block partial sum, fp32 accumulation, a
// 64-expanded-row window), re-planned for one GB300 SM per CTA:
//  * every CTA routes the (at most 64) expanded rows itself, so all CTAs hold
//    the same maps and no launch sits between the call and the weight stream;
//  * a unit is 16*RGS k rows x NT columns of one active expert's weights
//    (32 KB when NT/8 * RGS = 512).  The units of all active experts are laid
//    end to end (expert slot, column tile, k) and cut into one range per CTA
//    of equal cost ("stream-K"); a CTA's units of one (expert, tile) pair form
//    a segment, which it reduces to fp32 partial rows in the workspace;
//  * all rows of an expert are decoded in one pass over its units (up to
//    kMaxRC rows at once, more rows in chunks), so each weight byte is read
//    from HBM once and converted once per chunk;
//  * warp 16 copies the units (cp.async.bulk into a 4-slot ring, evict-first,
//    the unit's k-major scale rows in the same slot), FC1's and then FC2's
//    without waiting in between; warp 17 stages each window of activations as
//    fp16 rows rescaled by a power of two per row (largest |x| in
//    [2^14, 2^15), so every bf16 value is exact in fp16), double-buffered
//    ahead of the 16 consumer warps;
//  * consumer thread (w, rg) owns column word w (8 columns) of k-group rg
//    (16 rows) of every unit: 16 LDS.32, the hardware cvt.rn.f16x2.e2m1x2,
//    fma.rn.f32.f16 (exact fp16 products, fp32 sums), the 16-row partial
//    scaled once by its block scale (NVFP4: hardware E4M3 -> f16 conversion;
//    MXFP4: 2^(b-127) by bit placement);
//  * a grid barrier separates FC1 from FC2; the CTA then computes the FC2
//    activations a = bf16(SwiGLU(g1 * sum of FC1 partials)) it needs into
//    shared memory, in one flat loop (all partial loads in flight at once);
//    after a second grid barrier out[t] = bf16(sum_j w[t][j] * g2 * sum of
//    FC2 partials of (t, j)).  Every sum runs in a fixed order: the result is
//    deterministic;
//  * cooperative launch (all CTAs resident); grid-barrier counters live in
//    the workspace header and the last CTA out returns them to zero, so a
//    call on a primed workspace chains by programmatic dependent launch;
//  * every wait is bounded: one that gives up sets the device error flag
//    (header word 1) and the CTA carries on without waiting again.
#include <algorithm>
#include <atomic>

#include "decode_common.cuh"

namespace qmoe {
namespace dk {

constexpr int kCons = 512;                 // consumer threads (16 warps)
constexpr int kConsWarps = kCons / 32;
constexpr int kThreads = kCons + 64;       // + the copy warp + the activation warp
constexpr int kWarpP = kConsWarps;         // weight copies
constexpr int kWarpH = kConsWarps + 1;     // activation windows
constexpr int kRing = 5;                   // weight ring slots (32 KB units)
constexpr int kMaxRC = 2;                  // rows decoded together (more rows: chunks of two)
constexpr int kWinElems = 2048;            // fp16 activations per window buffer (rows x window length)
constexpr int kPreElems = 4096;            // bf16 FC2 activations computed per group
constexpr int kMaxSlots = 64;
constexpr int kMaxPairs = 512;             // (slot, tile) pairs whose CTA range is tabulated
constexpr int kHoldPairs = 128;            // pairs whose holders' partial-row bases are tabulated
constexpr int kMaxCtas = 256;
constexpr int kSmemOptin = 232448;
constexpr uint32_t kWaitLimit = 1u << 22;
constexpr uint32_t kSpinLimit = 1u << 24;

struct Shared {
  uint64_t full[kRing], empty[kRing];  // weight ring
  uint64_t xfull[2], xempty[2];        // activation windows
  uint64_t pre_ready;                  // an FC2 activation group is in place (every consumer thread arrives)
  uint64_t tables_ready;               // the cross-CTA lookup tables are in place (every lane of the activation warp)
  int4 slot[kMaxSlots];                // {expert, first permuted row, rows, 0}, ascending expert
  int row_tok[kMaxSlots], row2slot[kMaxSlots];
  int r_ids[kMaxSlots], r_e2p[kMaxSlots], r_p2e[kMaxSlots];
  float r_w[kMaxSlots];
  float gs[2][kMaxSlots];              // global scales per slot
  int scum[2][kMaxSlots + 1];          // split cost prefix over the slots
  int bnd[2][kMaxCtas + 1];            // unit range of each CTA
  int offp[2][kMaxCtas + 1];           // first partial row of each CTA's region (c * cap) minus the partial
                                       // rows of the pairs before its first pair; -1 for a CTA without units
  uint32_t pr[2][kMaxPairs];           // first | last CTA << 16 holding units of each (slot, tile) pair
  alignas(16) int hold[2][kHoldPairs][8];  // partial-row base (row 0) in the regions of the first 8 CTAs
                                       // holding each pair, in CTA order; -1: none
  int win_sh[2][kMaxRC];               // row shifts of the window in each buffer
  int na;
  int abort;
};

// ---- work split -------------------------------------------------------------------------

__device__ __forceinline__ int nchunks(int rows) { return (rows + kMaxRC - 1) / kMaxRC; }
// cost of one unit of an r-row expert and of a whole (expert, tile) pair, in
// the plan's units (a 32 KB unit decoded for one row is u0 + u1)
__device__ __forceinline__ int unit_cost(const DkFc &F, int rows) { return nchunks(rows) * F.u0 + rows * F.u1; }
__device__ __forceinline__ int pair_cost(const DkPlan &P, const DkFc &F, int rows) {
  return nchunks(rows) * P.pass + F.ku * unit_cost(F, rows);
}
// partial rows of all pairs before pair p = (slot a, tile t)
__device__ __forceinline__ int wpair(const Shared &S, const DkFc &F, int p) {
  const int a = p / F.ct, t = p - a * F.ct;
  return F.ct * S.slot[a].y + t * S.slot[a].z;
}
__device__ __forceinline__ int rows_of_pair(const Shared &S, const DkFc &F, int p) { return S.slot[p / F.ct].z; }

// first unit of CTA c: the first unit that starts at or after c * total / G
__device__ int split_bound(const Shared &S, const DkPlan &P, int f, int c, int G) {
  const DkFc &F = P.f[f];
  const int na = S.na;
  if (c >= G) return na * F.ct * F.ku;
  const long long total = S.scum[f][na];
  const long long x = total * c / G;
  int lo = 0, hi = na - 1;  // the last slot whose prefix is <= x
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (S.scum[f][mid] <= x) lo = mid; else hi = mid - 1;
  }
  const int r = S.slot[lo].z, cu = unit_cost(F, r), pc = pair_cost(P, F, r);
  const long long rem = x - S.scum[f][lo];
  const int q = (int)(rem / pc);
  int u;
  if (q >= F.ct) {
    u = F.ct * F.ku;
  } else {
    const long long v = rem - (long long)q * pc - (long long)nchunks(r) * P.pass;
    u = q * F.ku + (v <= 0 ? 0 : (int)min((long long)F.ku, (v + cu - 1) / cu));
  }
  return lo * F.ct * F.ku + u;
}
// CTA holding unit u: the largest c with bnd[c] <= u
__device__ __forceinline__ int cta_of(const int *bnd, int u) {
  int lo = 0, hi = (int)gridDim.x - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (bnd[mid] <= u) lo = mid; else hi = mid - 1;
  }
  return lo;
}
// partial rows CTA c writes for FC f (one row set per segment)
__device__ __forceinline__ int rows_written(const Shared &S, const DkFc &F, int f, int c) {
  const int lo = S.bnd[f][c], hi = S.bnd[f][c + 1];
  if (lo >= hi) return 0;
  const int p0 = lo / F.ku, p1 = (hi - 1) / F.ku;
  return wpair(S, F, p1) + rows_of_pair(S, F, p1) - wpair(S, F, p0);
}
// Partial rows: CTA c owns rows [c * cap, (c + 1) * cap) of FC f's partial
// array (cap from the plan bounds the rows any CTA writes); its segments'
// row sets follow one another there.  offp(c) = c * cap - wpair(first pair of c).
__device__ __forceinline__ int offp_of(const Shared &S, const DkFc &F, int f, int c) {
  const int lo = S.bnd[f][c];
  return lo < S.bnd[f][c + 1] ? c * F.cap - wpair(S, F, lo / F.ku) : -1;
}
// first and last CTA holding units of pair p
__device__ __forceinline__ void pair_ctas(const Shared &S, const DkFc &F, int f, int p, int &cf, int &cl) {
  if (p < kMaxPairs) {
    const uint32_t v = S.pr[f][p];
    cf = (int)(v & 0xFFFFu);
    cl = (int)(v >> 16);
  } else {
    cf = cta_of(S.bnd[f], p * F.ku);
    cl = cta_of(S.bnd[f], p * F.ku + F.ku - 1);
  }
}

// ---- the (segment, row chunk, window) sequence every role walks ---------------------------

// A window: rows [c0, c0 + rc) of segment (pair p = slot a, tile t; units
// [j0, j1) of the pair), units [wj0, wj1), k range [k0, k0 + klen).  RC is rc
// rounded up to a power of two; WL = kWinElems / RC activations per row.
struct Cur {
  int f, hi, nextu;
  int p, a, t, rows, j0, j1;
  int c0, rc, RC, WL, wu;
  int wj0, wj1, k0, klen;
  bool valid;
};

__device__ __forceinline__ void win_set(Cur &c, const DkFc &F) {
  c.wj1 = min(c.j1, c.wj0 + c.wu);
  c.k0 = c.wj0 * F.UK;
  c.klen = min(F.K, c.wj1 * F.UK) - c.k0;
}
__device__ __forceinline__ void chunk_start(Cur &c, const DkFc &F) {
  c.rc = min(kMaxRC, c.rows - c.c0);
  c.RC = c.rc <= 1 ? 1 : 2;
  c.WL = kWinElems / c.RC;
  c.wu = c.WL / F.UK;
  c.wj0 = c.j0;
  win_set(c, F);
}
__device__ __forceinline__ void seg_start(Cur &c, const Shared &S, const DkFc &F) {
  const int u = c.nextu;
  if (u >= c.hi) {
    c.valid = false;
    return;
  }
  c.p = u / F.ku;
  c.a = c.p / F.ct;
  c.t = c.p - c.a * F.ct;
  c.j0 = u - c.p * F.ku;
  c.j1 = min(c.hi - c.p * F.ku, F.ku);
  c.nextu = c.p * F.ku + c.j1;
  c.rows = S.slot[c.a].z;
  c.c0 = 0;
  c.valid = true;
  chunk_start(c, F);
}
__device__ __forceinline__ void cur_begin(Cur &c, const Shared &S, const DkPlan &P, int f, int lo, int hi) {
  c.f = f;
  c.nextu = lo;
  c.hi = hi;
  seg_start(c, S, P.f[f]);
}
__device__ __forceinline__ void cur_begin(Cur &c, const Shared &S, const DkPlan &P, int f) {
  cur_begin(c, S, P, f, S.bnd[f][blockIdx.x], S.bnd[f][blockIdx.x + 1]);
}
// advance to the next window (the next row chunk, the next segment, or invalid)
__device__ __forceinline__ void cur_next(Cur &c, const Shared &S, const DkPlan &P) {
  const DkFc &F = P.f[c.f];
  c.wj0 = c.wj1;
  if (c.wj0 < c.j1) {
    win_set(c, F);
    return;
  }
  c.c0 += kMaxRC;
  if (c.c0 < c.rows) {
    chunk_start(c, F);
    return;
  }
  seg_start(c, S, F);
}
// FC2 activation groups: consecutive windows whose bf16 activations fit in
// kPreElems together.  Returns true when window c opens a new group (and
// sets its offset in the group buffer).
__device__ __forceinline__ bool group_step(const Cur &c, int &used, int &off) {
  const int sz = c.rc * c.klen;
  const bool fresh = used < 0 || used + sz > kPreElems;
  if (fresh) used = 0;
  off = used;
  used += sz;
  return fresh;
}

// ---- waits ------------------------------------------------------------------------------------

__device__ __forceinline__ bool wait_bar(Shared &S, const LayerArgs &g, uint64_t *bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint32_t limit = *(volatile int *)&S.abort ? 64u : kWaitLimit;
  for (uint32_t i = 0; i < limit; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  *(volatile int *)&S.abort = 1;
  // the flag keeps the first failure: 100 + the barrier's index in the shared block
  atomicCAS(g.meta + 1, 0, 100 + (int)(bar - reinterpret_cast<uint64_t *>(&S)));
  return false;
}

__device__ __forceinline__ void cons_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kCons) : "memory"); }

// One thread per CTA arrives (release) and polls (acquire); one poller per
// CTA keeps the counter's L2 slice free for the arrivals.
__device__ __noinline__ void grid_barrier(Shared &S, const LayerArgs &g, int32_t *ctr) {
  cons_sync();
  if (threadIdx.x == 0) {
    asm volatile("red.release.gpu.global.add.s32 [%0], 1;" ::"l"(ctr) : "memory");
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

// The last CTA to leave returns both barrier counters and the exit counter to
// zero (each CTA's barrier thread calls this after its last acquire poll).
__device__ __forceinline__ void leave_counters(const LayerArgs &g) {
  if (atomicAdd(g.meta + 4, 1) == (int)gridDim.x - 1) {
    atomicExch(g.meta + 2, 0);
    atomicExch(g.meta + 3, 0);
    atomicExch(g.meta + 4, 0);
  }
}

// ---- the weight-copy warp ------------------------------------------------------------------------

template <int FMT>
__device__ __noinline__ void producer(Shared &S, const LayerArgs &g, const DkPlan &P, unsigned char *ring,
                                      int4 range) {
  constexpr int BS = FMT == QMOE_NVFP4 ? kNvfp4Block : kMxfp4Block;
  const int lane = (int)lane_id();
  const uint64_t pol = l2_evict_first_policy();
  uint32_t it = 0;
  uint32_t last_it[kRing];
#pragma unroll
  for (int s = 0; s < kRing; ++s) last_it[s] = ~0u;

  for (int f = 0; f < 2; ++f) {
    const DkFc &F = P.f[f];
    const uint8_t *wbase = f == 0 ? g.w1 : g.w2;
    const uint8_t *sbase = f == 0 ? g.s1 : g.s2;
    Cur c;
    for (cur_begin(c, S, P, f, f == 0 ? range.x : range.z, f == 0 ? range.y : range.w); c.valid; cur_next(c, S, P)) {
      const int e = S.slot[c.a].x;
      const uint8_t *wexp = wbase + (size_t)e * F.K * (F.N / 2) + (size_t)c.t * F.row_bytes;
      const uint8_t *sexp = sbase + (size_t)e * F.nblocks * F.N + (size_t)c.t * F.NT;
      for (int j = c.wj0; j < c.wj1; ++j, ++it) {
        const int s = (int)(it % kRing);
        if (it >= (uint32_t)kRing) {
          int ok = 1;
          if (lane == 0) ok = wait_bar(S, g, &S.empty[s], ((it / kRing) + 1u) & 1u) ? 1 : 0;
          if (!__shfl_sync(0xFFFFFFFFu, ok, 0)) goto drain;
        }
        last_it[s] = it;
        unsigned char *dst = ring + (size_t)s * P.slot_bytes;
        const int r0 = j * F.UK, nr = min(F.UK, F.K - r0);
        const int b0 = r0 / BS, nbu = min(F.bpu, F.nblocks - b0);
        if (lane == 0) mbar_expect_tx(&S.full[s], (uint32_t)(nr * F.row_bytes + nbu * F.NT));
        __syncwarp();
        // the slot was only read by generic loads of the consumers before they
        // released it: no proxy fence is needed before the copy writes it
        if (F.ct == 1) {  // contiguous unit: one copy per row group, one for the scale rows
          for (int q = lane; q < F.RGS; q += 32) {
            const int n16 = min(16, nr - 16 * q);
            if (n16 > 0)
              bulk_g2s_stream(dst + (size_t)q * F.rg_stride, wexp + (size_t)(r0 + 16 * q) * F.row_bytes,
                              (uint32_t)(n16 * F.row_bytes), &S.full[s], pol);
          }
          if (lane == 31)
            bulk_g2s_stream(dst + F.sc_off, sexp + (size_t)b0 * F.N, (uint32_t)(nbu * F.NT), &S.full[s], pol);
        } else {
          // a column tile of the unit: one 2-D tensor copy (16 rows x row_bytes)
          // per row group; one bulk copy per row would serialise in the copy
          // engine (a fixed cost per copy, ~32 per unit)
          const CUtensorMap *map = f == 0 ? &g.tm_w1 : &g.tm_w2;
          for (int q = lane; q < F.RGS; q += 32)
            if (16 * q < nr)
              tensor_g2s_2d(dst + (size_t)q * F.rg_stride, map, c.t * (F.row_bytes / 4), e * F.K + r0 + 16 * q,
                            &S.full[s]);
          for (int b = lane; b < nbu; b += 32)
            bulk_g2s_stream(dst + F.sc_off + (size_t)b * F.NT, sexp + (size_t)(b0 + b) * F.N, (uint32_t)F.NT,
                            &S.full[s], pol);
        }

      }
    }
  }
drain:
  // no CTA exits while its own copies still land in its shared memory: wait
  // (bounded, even after an abort) for the last copy issued into each slot
  if (lane == 0) {
    for (int s = 0; s < kRing; ++s) {
      if (last_it[s] == ~0u) continue;
      uint32_t i = 0;
      while (!mbar_try_wait(&S.full[s], (last_it[s] / kRing) & 1u) && ++i < kWaitLimit) {
      }
    }
  }
  __syncwarp();
}


// ---- the activation warp -----------------------------------------------------------------------

// Window c into buffer b (`win`): rows [c0, c0 + rc) of its k range as fp16,
// each row scaled by 2^-sh, sh putting its largest |value| in [2^14, 2^15)
// (so every bf16 value is exact in fp16); the shifts go to win_sh[b].  FC1
// reads the token rows of x, FC2 the rows (klen bf16 each) of its group at `pre`.
__device__ __forceinline__ void stage_window(Shared &S, const LayerArgs &g, const Cur &c, const uint16_t *pre, int b,
                                          __half *win) {
  const int lane = (int)lane_id();
  const int nv = c.klen >> 3;  // 8-value vectors per row (klen is a multiple of 16)
  for (int rr = 0; rr < c.rc; ++rr) {
    const uint16_t *src = c.f == 0 ? g.x + (size_t)S.row_tok[S.slot[c.a].y + c.c0 + rr] * g.H + c.k0
                                   : pre + (size_t)rr * c.klen;
    uint32_t m = 0;
    for (int q = lane; q < nv; q += 32) m = max(m, absmax_bf16x8(*reinterpret_cast<const uint4 *>(src + 8 * q)));
    m = __reduce_max_sync(0xFFFFFFFFu, m);
    const int sh = row_shift(m);
    const float fsc = pow2f(-sh);
    uint4 *dst = reinterpret_cast<uint4 *>(win + (size_t)rr * c.WL);
    for (int q = lane; q < nv; q += 32) dst[q] = bf16x8_to_f16x8(*reinterpret_cast<const uint4 *>(src + 8 * q), fsc);
    if (lane == 0) S.win_sh[b][rr] = sh;
  }
}

// Lookup tables of the cross-CTA sums (needed once the FC1 partials are
// complete), by the activation warp once its FC1 windows are staged (off the
// consumers' path): every CTA's partial-row offset, the CTA range of every
// (slot, tile) pair, the holders' partial-row bases of the tabulated pairs
// and the slots' global scales.  The consumers wait for them (tables_ready)
// after the first grid barrier.
__device__ __noinline__ void build_tables(Shared &S, const LayerArgs &g, const DkPlan &P) {
  const int lane = (int)lane_id(), G = (int)gridDim.x, na = S.na;
  const int np0 = min(na * P.f[0].ct, kMaxPairs), np1 = min(na * P.f[1].ct, kMaxPairs);
  for (int i = lane; i < 2 * G + np0 + np1 + na; i += 32) {
    if (i < 2 * G) {
      const int f = i >= G ? 1 : 0, c = i - f * G;
      S.offp[f][c] = offp_of(S, P.f[f], f, c);
    } else if (i < 2 * G + np0 + np1) {
      const int f = i >= 2 * G + np0 ? 1 : 0, p = i - 2 * G - (f ? np0 : 0);
      const DkFc &F = P.f[f];
      const int cf = cta_of(S.bnd[f], p * F.ku), cl = cta_of(S.bnd[f], p * F.ku + F.ku - 1);
      S.pr[f][p] = (uint32_t)cf | ((uint32_t)cl << 16);
      if (p < kHoldPairs) {
        const int wp = wpair(S, F, p);
        for (int u = 0; u < 8; ++u) {
          const int o = cf + u <= cl ? offp_of(S, F, f, cf + u) : -1;
          S.hold[f][p][u] = o >= 0 ? o + wp : -1;
        }
        if (cl - cf >= 8) S.hold[f][p][7] = -2;  // more than 8 holders: not tabulated
      }
    } else {
      const int a = i - 2 * G - np0 - np1;
      S.gs[0][a] = g.g1 ? __ldg(g.g1 + S.slot[a].x) : 1.0f;
      S.gs[1][a] = g.g2 ? __ldg(g.g2 + S.slot[a].x) : 1.0f;
    }
  }
  mbar_arrive(&S.tables_ready);  // every lane, after its own stores
}

__device__ __noinline__ void warm_code(Shared &S, const LayerArgs &g, const DkPlan &P, uint16_t *pre);

__device__ __noinline__ void activations(Shared &S, const LayerArgs &g, const DkPlan &P, __half *wins,
                                         const uint16_t *pre) {
  const int lane = (int)lane_id();
  uint32_t wn = 0, gidx = 0;
  int gused = -1;
  for (int f = 0; f < 2; ++f) {
    if (f == 1) {  // every FC1 window is staged
      build_tables(S, g, P);
      warm_code(S, g, P, const_cast<uint16_t *>(pre));
    }
    Cur c;
    for (cur_begin(c, S, P, f); c.valid; cur_next(c, S, P), ++wn) {
      const uint16_t *src = nullptr;
      if (f == 1) {
        int goff;
        if (group_step(c, gused, goff)) {  // the consumers compute each group after the first grid barrier
          if (lane == 0) wait_bar(S, g, &S.pre_ready, gidx & 1u);
          __syncwarp();
          ++gidx;
        }
        src = pre + goff;
      }
      const int b = (int)(wn & 1u);
      if (wn >= 2u) {
        if (lane == 0) wait_bar(S, g, &S.xempty[b], ((wn >> 1) + 1u) & 1u);
        __syncwarp();
      }
      stage_window(S, g, c, src, b, wins + (size_t)b * kWinElems);
      mbar_arrive(&S.xfull[b]);  // every lane, after its own stores
    }
  }
}

// ---- consumers -----------------------------------------------------------------------------------

// One k-group (16 k rows x the 8 columns of a word) of a unit for RC
// activation rows: the 16 words first, then per row pair of k the two decoded
// words times the fp16 activation pair; the 16-row partial is multiplied once
// by its block scale.  RC == 1 runs two independent FMA chains per column.
template <int FMT, int RC>
__device__ __forceinline__ void kgroup(const unsigned char *wp, int rb, const __half *xp, int xs, uint2 sv,
                                       float (&acc)[RC][8]) {
  if constexpr (RC == 1) {
    float sc[8];
    block_scales8<FMT>(sv, sc);
    uint32_t wv[16];
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) wv[kk] = *reinterpret_cast<const uint32_t *>(wp + (size_t)kk * rb);
    const uint4 xa = *reinterpret_cast<const uint4 *>(xp), xc = *reinterpret_cast<const uint4 *>(xp + 8);
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
  } else {
    float bp[RC][8];
#pragma unroll
    for (int r = 0; r < RC; ++r)
#pragma unroll
      for (int c = 0; c < 8; ++c) bp[r][c] = 0.f;
    // words loaded a pair at a time (RC rows of partial sums hold the registers)
#pragma unroll
    for (int kk = 0; kk < 16; kk += 2) {
      uint32_t p[4], q[4];
      dec8(*reinterpret_cast<const uint32_t *>(wp + (size_t)kk * rb), p);
      dec8(*reinterpret_cast<const uint32_t *>(wp + (size_t)(kk + 1) * rb), q);
#pragma unroll
      for (int r = 0; r < RC; ++r)
        fma16(p, q, *reinterpret_cast<const uint32_t *>(xp + (size_t)r * xs + kk), bp[r]);
    }
    float sc[8];
    block_scales8<FMT>(sv, sc);
#pragma unroll
    for (int r = 0; r < RC; ++r)
#pragma unroll
      for (int c = 0; c < 8; ++c) acc[r][c] = fmaf(bp[r][c], sc[c], acc[r][c]);
  }
}

// The partial rows of (pair p, row) in the regions of the first 8 CTAs
// holding p, in CTA order: idx[u] (in rows of NT floats) and bit u of vmask
// when CTA cf + u holds units of p.  Entries without one point at the first
// holder's row (which always exists), so that every load can be issued
// unconditionally and all of them are in flight together.
__device__ __forceinline__ void pair_rows8(const Shared &S, const DkFc &F, int f, int p, int row, int (&idx)[8],
                                           uint32_t &vmask, int &cf, int &cl) {
  if (p < kHoldPairs && S.hold[f][p][7] != -2) {  // tabulated: two 16-byte shared loads
    const int4 h0 = *reinterpret_cast<const int4 *>(&S.hold[f][p][0]);
    const int4 h1 = *reinterpret_cast<const int4 *>(&S.hold[f][p][4]);
    const int hb[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
    vmask = 0;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      idx[u] = max(hb[u], 0) + row;
      vmask |= (hb[u] >= 0 ? 1u : 0u) << u;
    }
    cf = 0;
    cl = 7;  // no holders beyond the first 8 (pairs with more are not tabulated)
    return;
  }
  pair_ctas(S, F, f, p, cf, cl);
  const int wp = wpair(S, F, p) + row;
  int o[8];
#pragma unroll
  for (int u = 0; u < 8; ++u) o[u] = S.offp[f][min(cf + u, cl)];
  vmask = 0;
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const bool v = cf + u <= cl && o[u] >= 0;
    idx[u] = (v ? o[u] : o[0]) + wp;
    vmask |= (v ? 1u : 0u) << u;
  }
}

// Sum over the CTAs holding pair p of FC f of their partial values at
// (row, col) and (row, col + 1), in CTA order (deterministic).
__device__ __forceinline__ float2 pair_sum2(const Shared &S, const DkFc &F, int f, const float *part, int p, int row,
                                            int col) {
  int idx[8], cf, cl;
  uint32_t vm;
  pair_rows8(S, F, f, p, row, idx, vm, cf, cl);
  float2 v[8];
#pragma unroll
  for (int u = 0; u < 8; ++u) {  // predicated: only the CTAs that hold units of p
    v[u] = make_float2(0.f, 0.f);
    if ((vm >> u) & 1u) v[u] = __ldcg(reinterpret_cast<const float2 *>(part + (size_t)idx[u] * F.NT + col));
  }
  float2 h = make_float2(0.f, 0.f);
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    h.x += v[u].x;
    h.y += v[u].y;
  }
  if (cl - cf >= 8) {  // more than 8 CTAs hold the pair: the rest in order
    pair_ctas(S, F, f, p, cf, cl);
    const int wp = wpair(S, F, p) + row;
    for (int c = cf + 8; c <= cl; ++c) {
      const int o = S.offp[f][c];
      if (o >= 0) {
        const float2 w = __ldcg(reinterpret_cast<const float2 *>(part + (size_t)(o + wp) * F.NT + col));
        h.x += w.x;
        h.y += w.y;
      }
    }
  }
  return h;
}
__device__ __forceinline__ float pair_sum1(const Shared &S, const DkFc &F, int f, const float *part, int p, int row,
                                           int col) {
  int idx[8], cf, cl;
  uint32_t vm;
  pair_rows8(S, F, f, p, row, idx, vm, cf, cl);
  float v[8];
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    v[u] = 0.f;
    if ((vm >> u) & 1u) v[u] = __ldcg(part + (size_t)idx[u] * F.NT + col);
  }
  float h = 0.f;
#pragma unroll
  for (int u = 0; u < 8; ++u) h += v[u];
  if (cl - cf >= 8) {
    pair_ctas(S, F, f, p, cf, cl);
    const int wp = wpair(S, F, p) + row;
    for (int c = cf + 8; c <= cl; ++c) {
      const int o = S.offp[f][c];
      if (o >= 0) h += __ldcg(part + (size_t)(o + wp) * F.NT + col);
    }
  }
  return h;
}

// FC2 activation k of row `row` (within slot a): bf16(SwiGLU(g1 * h)) with h
// the FC1 outputs of the gate and linear columns, 2k and 2k + 1
// (interleaved) or k and I + k (concatenated).
__device__ __forceinline__ uint16_t fc2_activation(const Shared &S, const LayerArgs &g, const DkPlan &P, int a, int row,
                                                   int k) {
  const DkFc &F = P.f[0];
  float hg, hl;
  if (g.fusion == 2) {
    const int tg = k / F.NT, tl = (g.I + k) / F.NT;
    hg = pair_sum1(S, F, 0, g.p1, a * F.ct + tg, row, k - tg * F.NT);
    hl = pair_sum1(S, F, 0, g.p1, a * F.ct + tl, row, g.I + k - tl * F.NT);
  } else {
    const int t = (2 * k) / F.NT;
    const float2 h = pair_sum2(S, F, 0, g.p1, a * F.ct + t, row, 2 * k - t * F.NT);
    hg = h.x;
    hl = h.y;
  }
  const float g1 = S.gs[0][a];
  return (uint16_t)f32_to_bf16_rne(swiglu(hg * g1, hl * g1, g.alpha, g.beta, g.limit));
}

// The FC2 activations of the group of windows starting at c, into `pre`
// (window after window, rows of klen values), by every consumer thread; each
// thread then arrives on pre_ready.
__device__ __forceinline__ void prestage_body(Shared &S, const LayerArgs &g, const DkPlan &P, const Cur c0,
                                              uint16_t *pre, bool dry = false) {
  Cur q = c0;
  int base = 0;
  bool first = true;
  int i = dry ? (int)lane_id() : (int)threadIdx.x;  // this thread's next element of the group
  while (q.valid) {
    const int sz = q.rc * q.klen;
    if (!first && base + sz > kPreElems) break;  // the group rule of group_step
#pragma unroll 1
    for (; i < base + sz; i += kCons) {
      const int loc = i - base, rr = loc / q.klen;
      const uint16_t v = fc2_activation(S, g, P, q.a, q.c0 + rr, q.k0 + loc - rr * q.klen);
      if (dry) return;  // a dry run (see warm_code) stops after one element
      pre[i] = v;
    }
    base += sz;
    first = false;
    cur_next(q, S, P);
  }
  if (!dry) mbar_arrive(&S.pre_ready);
}
// out of line for the groups after the first (inside the chunk loop, rare);
// the first group is computed inline at the start of FC2, where few registers
// are live (no call, no saved registers)
__device__ __noinline__ void prestage_group(Shared &S, const LayerArgs &g, const DkPlan &P, const Cur c0,
                                            uint16_t *pre) {
  prestage_body(S, g, P, c0, pre);
}

// All windows of one row chunk of a segment (c on its first window; on return
// c is on the next chunk's first window, or invalid).
template <int FMT, int RC>
__device__ __forceinline__ void run_chunk(Shared &S, const LayerArgs &g, const DkPlan &P, Cur &c, unsigned char *ring,
                                       __half *wins, uint16_t *pre, uint32_t &slot, uint32_t &phase, uint32_t &wn,
                                       int &gused, bool &first_group_done) {
  constexpr int BS = FMT == QMOE_NVFP4 ? kNvfp4Block : kMxfp4Block;
  const DkFc &F = P.f[c.f];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int wpw = 32 >> F.lg_rgs;
  const int rg = lane >> (5 - F.lg_rgs), wl = lane & (wpw - 1);
  const int w = warp * wpw + wl;
  const bool active = w < F.NW;
  // this thread's k-group rg of a unit: its words, and its 8 scale bytes, at
  // fixed offsets of every slot
  const int sc0 = F.sc_off + ((rg * 16) / BS) * F.NT + 8 * w;
  const int wo0 = rg * F.rg_stride + 4 * w;
  const int f = c.f, seg_p = c.p, seg_c0 = c.c0, rc = c.rc;
  float acc[RC][8];
#pragma unroll
  for (int r = 0; r < RC; ++r)
#pragma unroll
    for (int cc = 0; cc < 8; ++cc) acc[r][cc] = 0.f;
  int sh[RC];
  bool first = true;
  do {
    if (f == 1) {
      int goff;
      if (group_step(c, gused, goff)) {
        if (first_group_done) first_group_done = false;  // computed before the chunk loop
        else prestage_group(S, g, P, c, pre);
      }
    }
    const int b = (int)(wn & 1u);
    wait_bar(S, g, &S.xfull[b], (wn >> 1) & 1u);
#pragma unroll
    for (int r = 0; r < RC; ++r) {
      const int nsh = r < rc ? S.win_sh[b][r] : 0;
      if (!first && nsh != sh[r]) {
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) acc[r][cc] = ldexp2(acc[r][cc], sh[r] - nsh);
      }
      sh[r] = nsh;
    }
    first = false;
    const __half *xw = wins + (size_t)b * kWinElems;
    for (int j = c.wj0; j < c.wj1; ++j) {
      wait_bar(S, g, &S.full[slot], phase);
      const int kg = j * F.RGS + rg;
      const unsigned char *sb = ring + (size_t)slot * P.slot_bytes;
      if (active && kg < F.nkg)
        kgroup<FMT, RC>(sb + wo0, F.row_bytes, xw + (kg * 16 - c.k0), c.WL, *reinterpret_cast<const uint2 *>(sb + sc0),
                        acc);
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.empty[slot]);
      if (++slot == (uint32_t)kRing) {
        slot = 0;
        phase ^= 1u;
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.xempty[b]);
    ++wn;
    cur_next(c, S, P);
  } while (c.valid && c.p == seg_p && c.c0 == seg_c0);
  // combine the row groups (fixed butterfly) and write the partial rows
  for (int m = wpw; m < 32; m <<= 1)
#pragma unroll
    for (int r = 0; r < RC; ++r)
#pragma unroll
      for (int cc = 0; cc < 8; ++cc) acc[r][cc] += __shfl_xor_sync(0xFFFFFFFFu, acc[r][cc], m);
  if (active && rg == 0) {
    float *part = f == 0 ? g.p1 : g.p2;
    const int own_off = offp_of(S, F, f, (int)blockIdx.x), seg_row = wpair(S, F, seg_p) + seg_c0;
#pragma unroll
    for (int r = 0; r < RC; ++r) {
      if (r < rc) {
        // the sum is near the rescaled row's magnitude, so undoing 2^-sh cannot underflow
        const float un = pow2f(sh[r]);
        float4 *d = reinterpret_cast<float4 *>(part + (size_t)(own_off + seg_row + r) * F.NT + 8 * w);
        d[0] = make_float4(acc[r][0] * un, acc[r][1] * un, acc[r][2] * un, acc[r][3] * un);
        d[1] = make_float4(acc[r][4] * un, acc[r][5] * un, acc[r][6] * un, acc[r][7] * un);
      }
    }
  }
}

// out[t][n] = bf16(sum_j w[t][j] * g2 * y_j[n]) once every FC2 partial is
// written: 8 lanes per column pair, lane j gathers expert j's FC2 partials;
// the lanes are summed by a fixed butterfly.
__device__ __noinline__ void finalize(Shared &S, const LayerArgs &g, const DkPlan &P, bool dry = false) {
  const DkFc &F = P.f[1];
  const int half = g.H / 2;
  const int items = g.T * half * 8;
  const int items_pad = (items + 31) & ~31;
  const int i0 = dry ? (int)lane_id() : (int)blockIdx.x * kCons + (int)threadIdx.x;
  for (int idx = i0; idx < items_pad; idx += (int)gridDim.x * kCons) {
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
      const int t2 = n / F.NT;
      const float2 s = pair_sum2(S, F, 1, g.p2, a * F.ct + t2, p - S.slot[a].y, n - t2 * F.NT);
      const float wgt = S.r_w[ex], g2 = S.gs[1][a];
      y0 = wgt * (s.x * g2);
      y1 = wgt * (s.y * g2);
    }
#pragma unroll
    for (int m = 4; m > 0; m >>= 1) {
      y0 += __shfl_xor_sync(0xFFFFFFFFu, y0, m);
      y1 += __shfl_xor_sync(0xFFFFFFFFu, y1, m);
    }
    if (dry) return;  // a dry run (see warm_code) stops after one item
    if (ok && j == 0)
      reinterpret_cast<uint32_t *>(g.out + (size_t)t * g.H)[n / 2] = f32_to_bf16_rne(y0) | (f32_to_bf16_rne(y1) << 16);
  }
}

// The code that runs right after the grid barriers (the FC2 activations and
// the weighted un-permute) runs once per launch, so its first execution pays
// for every instruction fetch.  The activation warp, idle during FC1, runs it
// once without side effects (one element each, nothing stored, no barrier
// arrival: the FC1 partials it reads are still being written and the result
// is dropped), which brings that code into the SM's instruction cache.
__device__ __noinline__ void warm_code(Shared &S, const LayerArgs &g, const DkPlan &P, uint16_t *pre) {
  Cur c;
  cur_begin(c, S, P, 1);
  if (c.valid) prestage_body(S, g, P, c, pre, true);
  finalize(S, g, P, true);
}

template <int FMT>
__device__ __noinline__ void consumer(Shared &S, const LayerArgs &g, const DkPlan &P, unsigned char *ring,
                                      __half *wins, uint16_t *pre) {
  const int tid = threadIdx.x;
  // this CTA's partial rows must fit in its region (the plan's bound)
  if (tid < 2 && rows_written(S, P.f[tid], tid, (int)blockIdx.x) > P.f[tid].cap) {
    *(volatile int *)&S.abort = 1;
    atomicCAS(g.meta + 1, 0, 301);  // more partial rows than a CTA's region holds
  }
  uint32_t slot = 0, phase = 0, wn = 0;
  int gused = -1;
  bool first_group_done = false;
  for (int f = 0; f < 2; ++f) {
    if (f == 1) {
      grid_barrier(S, g, g.meta + 2);  // every FC1 partial is written
      wait_bar(S, g, &S.tables_ready, 0u);
    }
    Cur c;
    cur_begin(c, S, P, f);
    if (f == 1 && c.valid) {  // the first FC2 activation group, while few registers are live
      prestage_body(S, g, P, c, pre);
      first_group_done = true;
    }
    while (c.valid) {
      if (c.RC == 1)
        run_chunk<FMT, 1>(S, g, P, c, ring, wins, pre, slot, phase, wn, gused, first_group_done);
      else
        run_chunk<FMT, 2>(S, g, P, c, ring, wins, pre, slot, phase, wn, gused, first_group_done);
    }
  }
  grid_barrier(S, g, g.meta + 3);  // every FC2 partial is written
  if (tid == 0) leave_counters(g);
  finalize(S, g, P);
}

template <int FMT>
__global__ void __launch_bounds__(kThreads, 1) moe_decode_kernel(const __grid_constant__ LayerArgs g,
                                                                   const __grid_constant__ DkPlan P) {
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ Shared S;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int i = 0; i < kRing; ++i) {
      mbar_init(&S.full[i], 1);
      mbar_init(&S.empty[i], kConsWarps);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&S.xfull[i], 32);  // every lane of the activation warp
      mbar_init(&S.xempty[i], kConsWarps);
    }
    mbar_init(&S.pre_ready, kCons);
    mbar_init(&S.tables_ready, 32);
    mbar_fence_init();
    S.abort = 0;
  }
  // Launched with programmatic dependent launch, the kernel may start while
  // the previous kernel of the stream still runs: nothing in global memory is
  // touched before its results are visible.  The next kernel cannot become
  // resident on an SM before this kernel's CTA there exits.
  pdl_wait();
  pdl_launch_dependents();
  // routing, in every CTA with the routing kernel's top-k (bit-identical
  // experts in every CTA): warp w routes tokens w, w + 18, ...
  const int R = g.T * g.k;
  for (int t = warp; t < g.T; t += kThreads / 32) {
    if (g.route_n == 1) route_one_token<1>(g.logits, g.mix, t, g.E, g.k, g.normalize, S.r_ids, S.r_w);
    else if (g.route_n == 2) route_one_token<2>(g.logits, g.mix, t, g.E, g.k, g.normalize, S.r_ids, S.r_w);
    else if (g.route_n == 4) route_one_token<4>(g.logits, g.mix, t, g.E, g.k, g.normalize, S.r_ids, S.r_w);
    else route_one_token<8>(g.logits, g.mix, t, g.E, g.k, g.normalize, S.r_ids, S.r_w);
  }
  __syncthreads();
  {
    // the maps and the active-expert slots, then the split cost prefix of
    // both FCs over the slots: every warp computes them (and writes the same
    // values), so that no warp of the CTA idles at a barrier meanwhile
    RankOut o;
    o.e2p = S.r_e2p;
    o.p2e = S.r_p2e;
    o.row_tok = S.row_tok;
    o.row2slot = S.row2slot;
    o.slots = S.slot;
    o.na = &S.na;
    rank_rows_small(S.r_ids, R, g.E, g.k, o);
    __syncwarp();
    const int na = S.na, per = (na + 31) / 32;
#pragma unroll 1
    for (int f = 0; f < 2; ++f) {
      const DkFc &F = P.f[f];
      int sum = 0;
      for (int q = 0; q < per; ++q) {
        const int a = lane * per + q;
        if (a < na) sum += F.ct * pair_cost(P, F, S.slot[a].z);
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
        if (a < na) {
          S.scum[f][a] = run;
          run += F.ct * pair_cost(P, F, S.slot[a].z);
        }
      }
      if (lane == 31) S.scum[f][na] = run;
    }
  }
  if (blockIdx.x == 0 && g.ids_out && tid < R) g.ids_out[tid] = S.r_ids[tid];
  __syncthreads();
  if (S.na <= 0) return;  // every CTA sees the same count
  const int G = (int)gridDim.x;
  // 1 KB-aligned regions (the bulk copies need 16-byte alignment)
  unsigned char *base = smem + ((1024u - (smem_addr(smem) & 1023u)) & 1023u);
  unsigned char *ring = base;
  __half *wins = reinterpret_cast<__half *>(base + P.win_off);
  uint16_t *pre = reinterpret_cast<uint16_t *>(base + P.pre_off);
  if (warp == kWarpP) {
    // the copy warp computes its own unit ranges (lane l: FC l / 2, bound
    // blockIdx.x + l % 2) and starts the weight stream at once
    int bd = 0;
    if (lane < 4) bd = split_bound(S, P, lane >> 1, (int)blockIdx.x + (lane & 1), G);
    const int4 range = make_int4(__shfl_sync(0xFFFFFFFFu, bd, 0), __shfl_sync(0xFFFFFFFFu, bd, 1),
                                 __shfl_sync(0xFFFFFFFFu, bd, 2), __shfl_sync(0xFFFFFFFFu, bd, 3));
    producer<FMT>(S, g, P, ring, range);
    return;
  }
  {  // the unit ranges of every CTA, both FCs (one boundary per thread of the other nine warps)
    const int q = warp < kWarpP ? tid : tid - 32;
    for (int i = q; i <= 2 * G + 1; i += kThreads - 32) {
      if (i <= G) S.bnd[0][i] = split_bound(S, P, 0, i, G);
      else S.bnd[1][i - G - 1] = split_bound(S, P, 1, i - G - 1, G);
    }
  }
  asm volatile("bar.sync 2, %0;" ::"n"(kThreads - 32) : "memory");  // every warp but the copy warp
  if (warp == kWarpH) activations(S, g, P, wins, pre);
  else consumer<FMT>(S, g, P, ring, wins, pre);
}

}  // namespace dk

// ---- host side -------------------------------------------------------------------------------------

// Geometry of one FC: whole rows when that keeps at least half the consumer
// threads busy (NT / 8 column words x RGS row groups <= 512), else the widest
// column tile that keeps 7/8 of them busy, else the tiling with the most busy
// threads; unit = 16 * RGS k rows (one k-group per thread).
static bool make_dk_fc(int K, int N, int BS, DkFc &F) {
  int best = 0;
  F = DkFc{};
  for (int ct = 1; ct <= 64 && best < dk::kCons * 7 / 8; ++ct) {
    if (N % ct) continue;
    const int NT = N / ct;
    if (NT % 32) continue;
    const int NW = NT / 8;
    if (NW > dk::kCons) continue;
    int RGS = 1;
    while (NW * RGS * 2 <= dk::kCons && RGS < 32) RGS *= 2;
    if (NW * RGS > best) {
      best = NW * RGS;
      F.ct = ct;
      F.NT = NT;
      F.NW = NW;
      F.RGS = RGS;
    }
    if (ct == 1 && best >= dk::kCons / 2) break;  // whole rows (one copy per row group) with half the threads busy
  }
  if (best == 0) return false;
  F.K = K;
  F.N = N;
  F.lg_rgs = 0;
  while ((1 << F.lg_rgs) < F.RGS) ++F.lg_rgs;
  F.UK = 16 * F.RGS;
  F.ku = (K + F.UK - 1) / F.UK;
  F.nkg = K / 16;
  F.nblocks = K / BS;
  F.bpu = F.UK / BS > 0 ? F.UK / BS : 1;
  F.row_bytes = F.NT / 2;
  // row groups of a ring slot: 16 rows plus a pad that puts the row groups
  // one warp reads (WPW words each) in different banks
  const int wpw = 32 / F.RGS;
  F.rg_stride = 16 * F.row_bytes + 16 * (wpw / 4 > 1 ? wpw / 4 : 1);
  // tensor-copied row groups (ct > 1) start on 128-byte boundaries
  if (F.ct > 1) F.rg_stride = (F.rg_stride + 127) & ~127;
  F.sc_off = F.RGS * F.rg_stride;  // the unit's k-major scale rows follow its row groups
  return true;
}

qmoe_status make_dk_plan(int fmt, int T, int H, int I, int E, int k, DkPlan &P, size_t &p1_floats,
                         size_t &p2_floats) {
  (void)E;
  const int BS = block_size(fmt);
  P = DkPlan{};
  if (!make_dk_fc(H, 2 * I, BS, P.f[0]) || !make_dk_fc(I, H, BS, P.f[1])) {
    set_error("no column tiling of N = %d / %d fits the decode kernel", 2 * I, H);
    return QMOE_ERR_UNSUPPORTED;
  }
  const size_t G = (size_t)num_sms();
  if (G > (size_t)dk::kMaxCtas) {
    set_error("the decode kernel supports at most %d SMs (this GPU has %zu)", dk::kMaxCtas, G);
    return QMOE_ERR_UNSUPPORTED;
  }
  int slot = 0;
  for (int f = 0; f < 2; ++f) slot = std::max(slot, P.f[f].sc_off + P.f[f].bpu * P.f[f].NT);
  P.slot_bytes = (slot + 1023) & ~1023;
  P.win_off = dk::kRing * P.slot_bytes;
  P.pre_off = P.win_off + 2 * dk::kWinElems * 2;
  P.smem = P.pre_off + dk::kPreElems * 2 + 1024;  // + room to align the base to 1 KB
  if (P.smem + (int)sizeof(dk::Shared) > dk::kSmemOptin) {
    set_error("the decode kernel's buffers do not fit in shared memory (N = %d / %d)", 2 * I, H);
    return QMOE_ERR_UNSUPPORTED;
  }
  // split costs: a 32 KB unit decoded for one row = u0 + u1 (the conversion
  // and the per-row multiply-adds), a row chunk's start = pass.  With few
  // units per CTA the weight stream's latency, not the decode, sets a CTA's
  // time, and a unit costs nearly the same whatever its rows.
  // FC2's weights are mostly in shared memory before its decode starts, so
  // its units always cost by their rows.
  const double n1 = (double)(T * k) * P.f[0].ct * P.f[0].ku / (double)num_sms();
  P.f[0].u0 = n1 < 16.0 ? 56 : 24;
  P.f[0].u1 = n1 < 16.0 ? 8 : 40;
  P.f[1].u0 = 24;
  P.f[1].u1 = 40;
  P.pass = 48;
  // Partial rows: a fixed region of cap rows per CTA.  A CTA's range spans at
  // most two pairs that it shares with others (at most rows_max rows each)
  // and pairs inside it, each of which costs at least ku * u1 per row; the
  // range costs at most total / G + 1 and the total at most ct * R times a
  // one-row pair's cost, so the inner pairs hold at most
  // ceil(ct * R * pc1 / (G * ku * u1)) + 1 rows.
  const size_t R = (size_t)T * k, rows_max = std::min<size_t>((size_t)T, R);
  for (int f = 0; f < 2; ++f) {
    DkFc &F = P.f[f];
    const double pc1 = (double)P.pass + (double)F.ku * (F.u0 + F.u1);
    const double inner = std::ceil((double)F.ct * (double)R * pc1 / ((double)G * F.ku * F.u1)) + 1.0;
    F.cap = (int)std::min<double>((double)R * F.ct, 2.0 * (double)rows_max + inner);
  }
  p1_floats = G * (size_t)P.f[0].cap * P.f[0].NT;
  p2_floats = G * (size_t)P.f[1].cap * P.f[1].NT;
  return QMOE_OK;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// One FC's packed weights as a 2-D array of 32-bit words, E*K rows of N/8
// words, box = one row group (16 rows) of a column tile (row_bytes / 4 words).
static cudaError_t encode_weight_map(CUtensorMap *m, const uint8_t *w, int E, const DkFc &F) {
  static std::atomic<EncodeTiledFn> fn{nullptr};
  EncodeTiledFn f = fn.load(std::memory_order_acquire);
  if (!f) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q);
    if (err != cudaSuccess || q != cudaDriverEntryPointSuccess || !p) {
      set_error("cuTensorMapEncodeTiled is not available");
      return err != cudaSuccess ? err : cudaErrorNotSupported;
    }
    f = reinterpret_cast<EncodeTiledFn>(p);
    fn.store(f, std::memory_order_release);
  }
  const cuuint64_t dims[2] = {(cuuint64_t)(F.N / 8), (cuuint64_t)E * (cuuint64_t)F.K};
  const cuuint64_t strides[1] = {(cuuint64_t)(F.N / 2)};
  const cuuint32_t box[2] = {(cuuint32_t)(F.row_bytes / 4), 16u};
  const cuuint32_t es[2] = {1, 1};
  const CUresult r = f(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<uint8_t *>(w), dims, strides, box, es,
                       CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_error("cuTensorMapEncodeTiled failed (%d)", (int)r);
    return cudaErrorInvalidValue;
  }
  return cudaSuccess;
}

template <int FMT>
static cudaError_t launch_dk_fmt(const LayerArgs &a, const DkPlan &P, bool pdl, cudaStream_t stream) {
  static std::atomic<int> smem_set[kMaxDevices], smem_ok[kMaxDevices];
  const int dev = current_device();
  if (dev < 0) return cudaErrorInvalidDevice;
  auto kfn = dk::moe_decode_kernel<FMT>;
  if (P.smem > smem_set[dev].load(std::memory_order_acquire)) {
    cudaError_t err = cudaFuncSetAttribute(kfn, cudaFuncAttributePreferredSharedMemoryCarveout,
                                           cudaSharedmemCarveoutMaxShared);
    if (err != cudaSuccess) return err;
    err = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, P.smem);
    if (err != cudaSuccess) return err;
    smem_set[dev].store(P.smem, std::memory_order_release);
  }
  if (P.smem != smem_ok[dev].load(std::memory_order_acquire)) {  // one CTA per SM, or the cooperative launch is refused
    int per_sm = 0;
    cudaError_t err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kfn, dk::kThreads, P.smem);
    if (err != cudaSuccess) return err;
    if (per_sm < 1) {
      cudaFuncAttributes fa{};
      cudaFuncGetAttributes(&fa, kfn);
      set_error("decode kernel does not fit on an SM: %d registers x %d threads, %zu + %d bytes shared memory",
                fa.numRegs, dk::kThreads, (size_t)fa.sharedSizeBytes, P.smem);
      return cudaErrorCooperativeLaunchTooLarge;
    }
    smem_ok[dev].store(P.smem, std::memory_order_release);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_sms());
  cfg.blockDim = dim3(dk::kThreads);
  cfg.dynamicSmemBytes = P.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kfn, a, P);
}

cudaError_t launch_dk(const LayerArgs &a, const DkPlan &P, bool pdl, cudaStream_t stream) {
  LayerArgs g = a;
  if (P.f[0].ct > 1) {
    const cudaError_t err = encode_weight_map(&g.tm_w1, g.w1, g.E, P.f[0]);
    if (err != cudaSuccess) return err;
  }
  if (P.f[1].ct > 1) {
    const cudaError_t err = encode_weight_map(&g.tm_w2, g.w2, g.E, P.f[1]);
    if (err != cudaSuccess) return err;
  }
  if (g.fmt == QMOE_NVFP4) return launch_dk_fmt<QMOE_NVFP4>(g, P, pdl, stream);
  return launch_dk_fmt<QMOE_MXFP4>(g, P, pdl, stream);
}

}  // namespace qmoe
