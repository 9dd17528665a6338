// Warp-level top-k softmax routing, shared by the routing kernel and the
// decode layer kernel (which routes its few tokens itself, with the same code,
// so both select identical experts), and two one-warp builders of the R <= 64
// permute maps: the routing kernel's (every expert's offset) and the layer
// kernel's (only the experts that received rows).
//
// "[CUDA] Cut the MoE routing prologue/epilogue cost for small-batch decode"
// (PR #31156): one token row per warp held in registers and a stable packed
// key, expert ranking with warp matches.  Ties: packed stable key =
// order-preserving fp32 bits of the logit (-0.0 folded onto +0.0) in the high
// word, (0xFFFF - expert) in the low word.  Selection here: each lane sorts its
// own keys, then k rounds of a warp-wide maximum (redux.sync) pick the k
// largest keys, which the pages' butterfly of bitonic top-N merges also
// yields (the keys are distinct, so the k largest are one set in one order).
#pragma once

#include "qmoe_common.cuh"

namespace qmoe {

__device__ __forceinline__ uint64_t route_key(float v, int idx) {
  uint32_t b = __float_as_uint(v);
  if (b == 0x80000000u) b = 0u;
  uint32_t ord = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  return ((uint64_t)ord << 32) | (uint32_t)(0xFFFFu - (uint32_t)idx);
}
__device__ __forceinline__ int key_expert(uint64_t key) { return (int)(0xFFFFu - (uint32_t)(key & 0xFFFFu)); }
__device__ __forceinline__ float key_logit(uint64_t key) {
  uint32_t ord = (uint32_t)(key >> 32);
  uint32_t b = (ord & 0x80000000u) ? (ord & 0x7FFFFFFFu) : ~ord;
  return __uint_as_float(b);
}

// Descending bitonic sort of N register-resident keys.
template <int N>
__device__ __forceinline__ void bitonic_sort_desc(uint64_t (&a)[N]) {
#pragma unroll
  for (int size = 2; size <= N; size <<= 1)
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1)
#pragma unroll
      for (int i = 0; i < N; ++i) {
        const int j = i ^ stride;
        if (j > i) {
          const bool desc = (i & size) == 0;
          const uint64_t x = a[i], y = a[j];
          if (desc ? (x < y) : (x > y)) { a[i] = y; a[j] = x; }
        }
      }
}

// Warp-wide maximum of an unsigned word (redux.sync, all 32 lanes).
__device__ __forceinline__ uint32_t warp_max_u32(uint32_t v) {
  uint32_t r;
  asm volatile("redux.sync.max.u32 %0, %1, 0xffffffff;" : "=r"(r) : "r"(v));
  return r;
}

// The k <= 8 largest keys of the warp, descending, in every lane.  Every lane
// sorts its N keys; each round takes the warp maximum of the lanes' leading
// keys (the maximum high word, then the maximum low word among the lanes whose
// high word is that maximum) and the lane that held it drops it.  Valid keys
// are distinct and nonzero (the low word holds 0xFFFF - expert), padding keys
// are zero, and k never exceeds the number of valid keys.
template <int N>
__device__ __forceinline__ void warp_topk_keys(uint64_t (&a)[N], int k, uint64_t (&top)[kMaxTopK]) {
  bitonic_sort_desc<N>(a);
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j) top[j] = 0ull;
  for (int j = 0; j < k; ++j) {  // k is the same in every lane
    const uint32_t hi = (uint32_t)(a[0] >> 32), lo = (uint32_t)a[0];
    const uint32_t mh = warp_max_u32(hi);
    const uint32_t ml = warp_max_u32(hi == mh ? lo : 0u);
    const uint64_t best = ((uint64_t)mh << 32) | ml;
#pragma unroll
    for (int q = 0; q < kMaxTopK; ++q)
      if (q == j) top[q] = best;
    if (hi == mh && lo == ml) {
#pragma unroll
      for (int i = 0; i + 1 < N; ++i) a[i] = a[i + 1];
      a[N - 1] = 0ull;
    }
  }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, m);
  return v;
}

// One warp routes token t: ids/weights for its k experts.  With mix (the
// operator's router_weights, [T, E], input 14 of "MoE and QMoE - CUDA
// Operator Documentation" §2.3) the logits only select and the weights are
// mix[t][id] gathered at the selected experts, renormalised over the k like
// the softmax weights when normalize is set.
template <int N>
__device__ __forceinline__ void route_one_token(const float *__restrict__ logits, const float *__restrict__ mix, int t,
                                                int E, int k, int normalize, int32_t *__restrict__ ids,
                                                float *__restrict__ weights, int32_t *ids_smem = nullptr) {
  const int lane = (int)lane_id();
  const float *row = logits + (size_t)t * E;
  float v[N];
  uint64_t key[N];
#pragma unroll
  for (int i = 0; i < N; ++i) {
    const int e = lane + 32 * i;
    const bool ok = e < E;
    v[i] = ok ? __ldg(row + e) : 0.f;
    key[i] = ok ? route_key(v[i], e) : 0ull;
  }
  uint64_t top[kMaxTopK];
  warp_topk_keys<N>(key, k, top);
  const float mx = key_logit(top[0]);
  float s = 0.f;  // softmax denominator over all E (not needed when the k weights are renormalised)
  if (!normalize && !mix) {
#pragma unroll
    for (int i = 0; i < N; ++i)
      if (lane + 32 * i < E) s += expf(v[i] - mx);
    s = warp_sum(s);
  }
  // selected experts, in key order
  float sel_sum = 0.f;
  float mine_e = 0.f;
  int mine_id = 0;
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j) {
    if (j < k) {
      const float ej = mix ? __ldg(mix + (size_t)t * E + key_expert(top[j])) : expf(key_logit(top[j]) - mx);
      sel_sum += ej;
      if (j == lane) { mine_e = ej; mine_id = key_expert(top[j]); }
    }
  }
  if (lane < k) {
    ids[(size_t)t * k + lane] = mine_id;
    if (ids_smem) ids_smem[t * k + lane] = mine_id;
    weights[(size_t)t * k + lane] = normalize ? mine_e / sel_sum : (mix ? mine_e : mine_e / s);
  }
}

// Maps for R <= 64 assignments, built by one warp with no block barrier: lane l
// holds assignments l and l + 32; __match_any_sync ranks each half, the first
// half's per-expert counts (shared memory) offset the second half's ranks, so
// the rank is stable; then an exclusive scan over the experts.
__device__ inline void build_maps_small(const int32_t *ids_s, int R, int E, const RouteOut &o, int32_t *cnt /* smem [E] */,
                                 int32_t *off /* smem [E] */) {
  const int lane = (int)lane_id();
  const unsigned lt = (1u << lane) - 1u;
  for (int e = lane; e < E; e += 32) cnt[e] = 0;
  __syncwarp();
  const int i0 = lane, i1 = lane + 32;
  const bool v0 = i0 < R, v1 = i1 < R;
  const int e0 = v0 ? ids_s[i0] : -1 - lane, e1 = v1 ? ids_s[i1] : -100 - lane;
  const bool ok0 = v0 && e0 >= 0 && e0 < E, ok1 = v1 && e1 >= 0 && e1 < E;
  const unsigned p0 = __match_any_sync(0xFFFFFFFFu, e0);
  const int r0 = __popc(p0 & lt);
  if (ok0 && (p0 & lt) == 0u) cnt[e0] = __popc(p0);
  __syncwarp();
  const unsigned p1 = __match_any_sync(0xFFFFFFFFu, e1);
  const int r1 = (ok1 ? cnt[e1] : 0) + __popc(p1 & lt);
  __syncwarp();
  if (ok1 && (p1 & lt) == 0u) cnt[e1] += __popc(p1);
  __syncwarp();
  // exclusive scan of the counts
  const int per = (E + 31) / 32;
  int sum = 0;
  for (int q = 0; q < per; ++q) {
    const int e = lane * per + q;
    if (e < E) sum += cnt[e];
  }
  int incl = sum;
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    const int a = __shfl_up_sync(0xFFFFFFFFu, incl, m);
    if (lane >= m) incl += a;
  }
  int run = incl - sum;
  for (int q = 0; q < per; ++q) {
    const int e = lane * per + q;
    if (e < E) {
      o.offsets[e] = run;
      off[e] = run;
      run += cnt[e];
    }
  }
  if (lane == 31) o.offsets[E] = run;
  __syncwarp();
  if (ok0) { const int p = off[e0] + r0; o.e2p[i0] = p; o.p2e[p] = i0; }
  if (ok1) { const int p = off[e1] + r1; o.e2p[i1] = p; o.p2e[p] = i1; }
}

// The layer kernel's maps of R <= 64 expanded rows, by one warp with no shared
// scratch.  The stable ranking (operator doc §1, permute by expert) puts
// assignment i (= t * k + j, expert e_i) at permuted row
//   p_i = #{ i' : e_i' < e_i, or e_i' = e_i and i' < i },
// i.e. the rank of the key e_i * 64 + i among all keys; the rows of expert e
// start at #{ i' : e_i' < e } and number #{ i' : e_i' = e }.  One pass over
// the R keys (a broadcast shuffle each) gives all three counts; the first row
// of each expert marks its slot, and a warp OR of those marks numbers the
// slots in expert order.  Same maps as build_maps_small.
struct RankOut {
  int32_t *e2p, *p2e;      // [R]
  int32_t *row_tok;        // [R] token of each permuted row
  int32_t *row2slot;       // [R] slot of each permuted row
  int4 *slots;             // [min(E, R)] {expert, first row, rows, 0}, ascending expert
  int *na;                 // number of slots
};
__device__ inline void rank_rows_small(const int32_t *ids_s, int R, int E, int k, const RankOut &o) {
  const int lane = (int)lane_id();
  constexpr int kNone = 0x7FFFFFFF;  // absent or invalid assignment: sorts last, never written
  const int i0 = lane, i1 = lane + 32;
  const bool v0 = i0 < R && (unsigned)ids_s[min(i0, R - 1)] < (unsigned)E;
  const bool v1 = i1 < R && (unsigned)ids_s[min(i1, R - 1)] < (unsigned)E;
  const int key0 = v0 ? ids_s[i0] * 64 + i0 : kNone, key1 = v1 ? ids_s[i1] * 64 + i1 : kNone;
  const int e0 = key0 >> 6, e1 = key1 >> 6;
  int rank0 = 0, rank1 = 0, lt0 = 0, lt1 = 0, le0 = 0, le1 = 0;
#pragma unroll 8
  for (int m = 0; m < 32; ++m) {
    const int a = __shfl_sync(0xFFFFFFFFu, key0, m), ea = a >> 6;
    rank0 += a < key0; lt0 += ea < e0; le0 += ea <= e0;
    rank1 += a < key1; lt1 += ea < e1; le1 += ea <= e1;
  }
  if (R > 32) {  // the same in every lane
#pragma unroll 8
    for (int m = 0; m < 32; ++m) {
      const int a = __shfl_sync(0xFFFFFFFFu, key1, m), ea = a >> 6;
      rank0 += a < key0; lt0 += ea < e0; le0 += ea <= e0;
      rank1 += a < key1; lt1 += ea < e1; le1 += ea <= e1;
    }
  }
  // first rows of the experts' groups, as a 64-bit mask over permuted rows
  const bool h0 = v0 && rank0 == lt0, h1 = v1 && rank1 == lt1;
  const uint64_t c = (h0 ? 1ull << rank0 : 0ull) | (h1 ? 1ull << rank1 : 0ull);
  const uint64_t heads = ((uint64_t)__reduce_or_sync(0xFFFFFFFFu, (uint32_t)(c >> 32)) << 32) |
                         __reduce_or_sync(0xFFFFFFFFu, (uint32_t)c);
  if (v0) {
    const int a = __popcll(heads & ((2ull << rank0) - 1ull)) - 1;
    o.e2p[i0] = rank0; o.p2e[rank0] = i0; o.row_tok[rank0] = i0 / k; o.row2slot[rank0] = a;
    if (h0) o.slots[a] = make_int4(e0, rank0, le0 - lt0, 0);
  }
  if (v1) {
    const int a = __popcll(heads & ((2ull << rank1) - 1ull)) - 1;
    o.e2p[i1] = rank1; o.p2e[rank1] = i1; o.row_tok[rank1] = i1 / k; o.row2slot[rank1] = a;
    if (h1) o.slots[a] = make_int4(e1, rank1, le1 - lt1, 0);
  }
  if (lane == 0) *o.na = __popcll(heads);
}

}  // namespace qmoe
