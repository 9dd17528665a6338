// Warp-level top-k softmax routing and the R <= 64 permute maps, shared by the
// routing kernel and the decode layer kernel (which routes its few tokens
// itself, with the same code, so both produce identical results).
//
// "[CUDA] Cut the MoE routing prologue/epilogue cost for small-batch decode"
// (PR #31156): one token row per warp held in registers, per-lane bitonic sort,
// butterfly of bitonic top-N merges (C[i] = max(A[i], B[N-1-i]), symmetric, so
// one shuffle per key), expert ranking with warp matches.  Ties: packed stable
// key = order-preserving fp32 bits of the logit (-0.0 folded onto +0.0) in the
// high word, (0xFFFF - expert) in the low word.
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

// Sorts a bitonic sequence of N keys descending.
template <int N>
__device__ __forceinline__ void bitonic_clean_desc(uint64_t (&a)[N]) {
#pragma unroll
  for (int stride = N >> 1; stride > 0; stride >>= 1)
#pragma unroll
    for (int i = 0; i < N; ++i) {
      const int j = i ^ stride;
      if (j > i && a[i] < a[j]) { const uint64_t t = a[i]; a[i] = a[j]; a[j] = t; }
    }
}

// After the call every lane holds the N largest keys of the warp, descending.
template <int N>
__device__ __forceinline__ void warp_bitonic_topn(uint64_t (&a)[N]) {
  bitonic_sort_desc<N>(a);
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    uint64_t b[N];
#pragma unroll
    for (int i = 0; i < N; ++i) b[i] = __shfl_xor_sync(0xFFFFFFFFu, a[i], m);
#pragma unroll
    for (int i = 0; i < N; ++i) a[i] = a[i] > b[N - 1 - i] ? a[i] : b[N - 1 - i];
    bitonic_clean_desc<N>(a);
  }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, m);
  return v;
}

// One warp routes token t: ids/weights for its k experts.
template <int N>
__device__ __forceinline__ void route_one_token(const float *__restrict__ logits, int t, int E, int k,
                                                int normalize, int32_t *__restrict__ ids,
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
  warp_bitonic_topn<N>(key);
  const float mx = key_logit(key[0]);
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < N; ++i)
    if (lane + 32 * i < E) s += expf(v[i] - mx);
  s = warp_sum(s);
  // selected experts, in key order
  float sel_sum = 0.f;
  float mine_e = 0.f;
  int mine_id = 0;
#pragma unroll
  for (int j = 0; j < N; ++j) {
    if (j < k) {
      const float ej = expf(key_logit(key[j]) - mx);
      sel_sum += ej;
      if (j == lane) { mine_e = ej; mine_id = key_expert(key[j]); }
    }
  }
  if (lane < k) {
    ids[(size_t)t * k + lane] = mine_id;
    if (ids_smem) ids_smem[t * k + lane] = mine_id;
    weights[(size_t)t * k + lane] = normalize ? mine_e / sel_sum : mine_e / s;
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
  // exclusive scan of the counts; the list of experts with rows
  const int per = (E + 31) / 32;
  int sum = 0, nact = 0;
  for (int q = 0; q < per; ++q) {
    const int e = lane * per + q;
    if (e < E) { sum += cnt[e]; nact += cnt[e] > 0; }
  }
  int incl = sum, iact = nact;
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    const int a = __shfl_up_sync(0xFFFFFFFFu, incl, m), b = __shfl_up_sync(0xFFFFFFFFu, iact, m);
    if (lane >= m) { incl += a; iact += b; }
  }
  int run = incl - sum, arun = iact - nact;
  for (int q = 0; q < per; ++q) {
    const int e = lane * per + q;
    if (e < E) {
      const int c = cnt[e];
      o.offsets[e] = run;
      off[e] = run;
      if (c > 0 && o.active) o.active[arun] = e;
      if (c > 0 && o.slots) o.slots[arun] = SlotDesc{e, run, c, 0};
      arun += c > 0;
      run += c;
    }
  }
  if (lane == 31) {
    o.offsets[E] = run;
    if (o.meta) o.meta[0] = arun;
  }
  __syncwarp();
  if (ok0) { const int p = off[e0] + r0; o.e2p[i0] = p; o.p2e[p] = i0; }
  if (ok1) { const int p = off[e1] + r1; o.e2p[i1] = p; o.p2e[p] = i1; }
}

}  // namespace qmoe
