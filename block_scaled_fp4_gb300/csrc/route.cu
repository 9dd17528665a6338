// Top-k softmax routing and permute-by-expert maps.
//
// "[CUDA] Cut the MoE routing prologue/epilogue cost for small-batch decode"
// (PR #31156) describes the design idea kept here: one token row per warp held
// entirely in registers (no shared memory, no block sort), and expert ranking
// with warp matches instead of per-thread radix counters.  The warp top-k
// (route_common.cuh) sorts each lane's keys and takes the k largest with k
// rounds of a warp maximum.  Ties are broken by a packed stable key: fp32
// logit (order-preserving bits, -0.0 folded onto +0.0) in the high word,
// (0xFFFF - expert) in the low word, so a larger key means a larger logit,
// then a lower expert index.
#include "route_common.cuh"

namespace qmoe {

template <int N>
__global__ void __launch_bounds__(256) route_topk_kernel(const float *__restrict__ logits,
                                                        const float *__restrict__ mix, int T, int E, int k,
                                                        int normalize, int32_t *__restrict__ ids,
                                                        float *__restrict__ weights) {
  const int warps = blockDim.x >> 5;
  const int t = blockIdx.x * warps + (int)(threadIdx.x >> 5);
  if (t < T) route_one_token<N>(logits, mix, t, E, k, normalize, ids, weights);
}

// Stable ranking of the R = T*k assignments by expert, done by one CTA.
// Warp w owns a contiguous segment of expanded indices; inside a segment 32
// assignments at a time are ranked with __match_any_sync (lanes choosing the
// same expert), per-warp per-expert counts go to shared memory, then each
// expert's count is prefixed over warps (segment order = expanded order, so
// the rank is stable), then over experts.
// Lanes of the warp whose key equals this lane's: one ballot for validity and
// one per key bit (keys < 2^nbits), ANDed.  An invalid lane matches only
// itself.  Same result as __match_any_sync over the valid keys, without the
// match instruction's long, throughput-bound latency.
__device__ __forceinline__ unsigned match_key(int key, bool valid, int nbits) {
  unsigned m = __ballot_sync(0xFFFFFFFFu, valid);
  for (int b = 0; b < nbits; ++b) {
    const bool bit = (key >> b) & 1;
    const unsigned bb = __ballot_sync(0xFFFFFFFFu, bit);
    m &= bit ? bb : ~bb;
  }
  return valid ? m : (1u << lane_id());
}

__device__ void build_maps(const int32_t *ids, int R, int E, int32_t *offsets, int32_t *p2e, int32_t *e2p,
                           int32_t *cnt /* smem [W][E] */, int32_t *tot /* smem [E+1] */) {
  const int W = blockDim.x >> 5, w = (int)(threadIdx.x >> 5), lane = (int)lane_id();
  for (int i = threadIdx.x; i < W * E; i += blockDim.x) cnt[i] = 0;
  __syncthreads();
  const int seg = (R + W - 1) / W;
  const int lo = w * seg, hi = min(R, lo + seg);
  int32_t *mycnt = cnt + w * E;
  // kNB rounds of 32 ids are loaded together (independent loads, one
  // latency), then ranked round by round
  constexpr int kNB = 8;
  const unsigned lt = (1u << lane) - 1u;
  int nbits = 0;  // bits of the largest expert index
  while ((1 << nbits) < E) ++nbits;
  for (int base = lo; base < hi; base += 32 * kNB) {
    int eid[kNB];
#pragma unroll
    for (int j = 0; j < kNB; ++j) {
      const int i = base + 32 * j + lane;
      eid[j] = i < hi ? ids[i] : -1;
    }
#pragma unroll
    for (int j = 0; j < kNB; ++j) {
      const int i = base + 32 * j + lane;
      const bool valid = i < hi && eid[j] >= 0 && eid[j] < E;
      const int e = valid ? eid[j] : 0;
      const unsigned peers = match_key(e, valid, nbits);  // invalid lanes match only themselves
      if (valid) e2p[i] = mycnt[e] + __popc(peers & lt);  // rank within this warp's segment
      __syncwarp();
      if (valid && (peers & lt) == 0u) mycnt[e] += __popc(peers);
      __syncwarp();
    }
  }
  __syncthreads();
  // per expert: exclusive prefix over warps
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = 0;
    for (int ww = 0; ww < W; ++ww) {
      const int c = cnt[ww * E + e];
      cnt[ww * E + e] = run;
      run += c;
    }
    tot[e] = run;
  }
  __syncthreads();
  // exclusive scan over experts (warp 0)
  if (w == 0) {
    const int per = (E + 31) / 32;
    int sum = 0;
    for (int q = 0; q < per; ++q) {
      const int e = lane * per + q;
      if (e < E) sum += tot[e];
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
        const int c = tot[e];
        offsets[e] = run;
        tot[e] = run;
        run += c;
      }
    }
    if (lane == 31) offsets[E] = run;
  }
  __syncthreads();
  for (int base = lo; base < hi; base += 32 * kNB) {
    int ev[kNB], rv[kNB];
#pragma unroll
    for (int j = 0; j < kNB; ++j) {
      const int i = base + 32 * j + lane;
      ev[j] = i < hi ? ids[i] : -1;
      rv[j] = i < hi ? e2p[i] : 0;
    }
#pragma unroll
    for (int j = 0; j < kNB; ++j) {
      const int i = base + 32 * j + lane;
      const int e = ev[j];
      if (i >= hi || e < 0 || e >= E) continue;
      const int pr = tot[e] + mycnt[e] + rv[j];
      e2p[i] = pr;
      p2e[pr] = i;
    }
  }
}

// Routing of up to kFusedRouteMaxTokens tokens in one CTA (warp per token),
// then the maps.
template <int N>
__global__ void __launch_bounds__(256) route_maps_fused_kernel(const float *__restrict__ logits, int T, int E,
                                                              int k, int normalize, RouteOut o) {
  extern __shared__ int32_t smem_i32[];
  const int W = blockDim.x >> 5, w = (int)(threadIdx.x >> 5);
  const int R = T * k;
  if (R <= 64) {
    int32_t *ids_s = smem_i32, *cnt = smem_i32 + 64, *off = cnt + E;
    for (int t = w; t < T; t += W) route_one_token<N>(logits, o.mix, t, E, k, normalize, o.ids, o.weights, ids_s);
    __syncthreads();
    if (w == 0) build_maps_small(ids_s, R, E, o, cnt, off);
    return;
  }
  for (int t = w; t < T; t += W) route_one_token<N>(logits, o.mix, t, E, k, normalize, o.ids, o.weights);
  __syncthreads();
  build_maps(o.ids, R, E, o.offsets, o.p2e, o.e2p, smem_i32, smem_i32 + W * E);
}

// Prefill routing, second step: one CTA of 1024 threads builds the maps.
__global__ void __launch_bounds__(1024) maps_kernel(int R, int E, RouteOut o) {
  extern __shared__ int32_t smem_i32[];
  const int W = blockDim.x >> 5;
  build_maps(o.ids, R, E, o.offsets, o.p2e, o.e2p, smem_i32, smem_i32 + W * E);
}

int route_keys_per_lane(int E, int k) {
  int n = 1;
  while (n * 32 < E) n <<= 1;
  while (n < k) n <<= 1;
  return n;
}

template <int N>
static cudaError_t launch_route_n(const float *logits, int T, int E, int k, int normalize, const RouteOut &o,
                                  cudaStream_t stream) {
  if (T <= kFusedRouteMaxTokens) {
    const int threads = 256, W = threads / 32;
    size_t smem = sizeof(int32_t) * ((size_t)W * E + E + 1);
    const size_t smem_small = sizeof(int32_t) * (64 + 2 * (size_t)E);
    if (smem_small > smem) smem = smem_small;
    route_maps_fused_kernel<N><<<1, threads, smem, stream>>>(logits, T, E, k, normalize, o);
    return cudaGetLastError();
  }
  const int warps = 8;
  route_topk_kernel<N><<<(T + warps - 1) / warps, warps * 32, 0, stream>>>(logits, o.mix, T, E, k, normalize,
                                                                            o.ids, o.weights);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  const int threads = 1024, W = threads / 32;
  const size_t smem = sizeof(int32_t) * ((size_t)W * E + E + 1);
  maps_kernel<<<1, threads, smem, stream>>>(T * k, E, o);
  return cudaGetLastError();
}

cudaError_t launch_route(const float *logits, int T, int E, int k, int normalize, const RouteOut &o,
                         cudaStream_t stream) {
  switch (route_keys_per_lane(E, k)) {
    case 1: return launch_route_n<1>(logits, T, E, k, normalize, o, stream);
    case 2: return launch_route_n<2>(logits, T, E, k, normalize, o, stream);
    case 4: return launch_route_n<4>(logits, T, E, k, normalize, o, stream);
    case 8: return launch_route_n<8>(logits, T, E, k, normalize, o, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace qmoe
