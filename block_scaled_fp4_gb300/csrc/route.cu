// Top-k softmax routing and permute-by-expert maps.
//
// "[CUDA] Cut the MoE routing prologue/epilogue cost for small-batch decode"
// (PR #31156) describes the design idea kept here: one token row per warp held
// entirely in registers, each lane bitonic-sorts its own keys, then the warp
// runs a butterfly of bitonic top-N merges where the merge rule
// C[i] = max(A[i], B[N-1-i]) is symmetric, so one shuffle per key leaves both
// partners with the same result (no shared memory, no barrier); and expert
// ranking with warp ballots/matches instead of per-thread radix counters.
// Ties are broken by a packed stable key: fp32 logit (order-preserving bits,
// -0.0 folded onto +0.0) in the high word, (0xFFFF - expert) in the low word,
// so a larger key means a larger logit, then a lower expert index.
#include <cuda_fp16.h>

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
                                                float *__restrict__ weights) {
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
    weights[(size_t)t * k + lane] = normalize ? mine_e / sel_sum : mine_e / s;
  }
}

template <int N>
__global__ void __launch_bounds__(256) route_topk_kernel(const float *__restrict__ logits, int T, int E, int k,
                                                        int normalize, int32_t *__restrict__ ids,
                                                        float *__restrict__ weights) {
  const int warps = blockDim.x >> 5;
  const int t = blockIdx.x * warps + (int)(threadIdx.x >> 5);
  if (t < T) route_one_token<N>(logits, t, E, k, normalize, ids, weights);
}

// Stable ranking of the R = T*k assignments by expert, done by one CTA.
// Warp w owns a contiguous segment of expanded indices; inside a segment 32
// assignments at a time are ranked with __match_any_sync (lanes choosing the
// same expert), per-warp per-expert counts go to shared memory, then each
// expert's count is prefixed over warps (segment order = expanded order, so
// the rank is stable), then over experts.
__device__ void build_maps(const int32_t *ids, int R, int E, int32_t *offsets, int32_t *p2e, int32_t *e2p,
                           int32_t *active, int32_t *meta, SlotDesc *slots, int32_t *cnt /* smem [W][E] */,
                           int32_t *tot /* smem [E+1] */) {
  const int W = blockDim.x >> 5, w = (int)(threadIdx.x >> 5), lane = (int)lane_id();
  for (int i = threadIdx.x; i < W * E; i += blockDim.x) cnt[i] = 0;
  __syncthreads();
  const int seg = (R + W - 1) / W;
  const int lo = w * seg, hi = min(R, lo + seg);
  int32_t *mycnt = cnt + w * E;
  for (int base = lo; base < hi; base += 32) {
    const int i = base + lane;
    const int eid = i < hi ? ids[i] : -1;
    const bool valid = i < hi && eid >= 0 && eid < E;
    const int e = valid ? eid : -1 - lane;  // invalid lanes never match anyone
    const unsigned peers = __match_any_sync(0xFFFFFFFFu, e);
    const unsigned lt = (1u << lane) - 1u;
    if (valid) e2p[i] = mycnt[e] + __popc(peers & lt);  // rank within this warp's segment
    __syncwarp();
    if (valid && (peers & lt) == 0u) mycnt[e] += __popc(peers);
    __syncwarp();
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
  // exclusive scan over experts (warp 0), plus the list of experts with rows
  if (w == 0) {
    const int per = (E + 31) / 32;
    int sum = 0, nact = 0;
    for (int q = 0; q < per; ++q) {
      const int e = lane * per + q;
      if (e < E) { sum += tot[e]; nact += tot[e] > 0; }
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
        const int c = tot[e];
        offsets[e] = run;
        tot[e] = run;
        if (c > 0 && active) active[arun] = e;
        if (c > 0 && slots) slots[arun] = SlotDesc{e, run, c, 0};
        arun += c > 0;
        run += c;
      }
    }
    if (lane == 31) {
      offsets[E] = run;
      if (meta) meta[0] = arun;
    }
  }
  __syncthreads();
  for (int i = lo + lane; i < hi; i += 32) {
    const int e = ids[i];
    if (e < 0 || e >= E) continue;
    const int p = tot[e] + mycnt[e] + e2p[i];
    e2p[i] = p;
    p2e[p] = i;
  }
}

// Per-token power-of-two rescale of the activations into fp16 for the decode
// GEMVs: x16 = x * 2^-s with the row's largest |x| * 2^-s in [2^14, 2^15), so
// every finite bf16 value keeps its 8 significant bits in fp16.  One warp per token.
__device__ void convert_token_fp16(const uint16_t *x, int H, int t, uint16_t *x16, int32_t *xshift) {
  const int lane = (int)lane_id();
  const uint16_t *row = x + (size_t)t * H;
  uint32_t m = 0;
  for (int i = lane * 8; i < H; i += 256) {
    const uint4 v = *reinterpret_cast<const uint4 *>(row + i);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) m = max(m, max(w[q] & 0x7FFFu, (w[q] >> 16) & 0x7FFFu));
  }
#pragma unroll
  for (int s = 16; s > 0; s >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, s));
  int sh = 0;
  if (m != 0u) sh = max(-100, min(100, (int)((m >> 7) & 0xFFu) - 127 - 14));
  const float f = __uint_as_float((uint32_t)(127 - sh) << 23);
  for (int i = lane * 8; i < H; i += 256) {
    const uint4 v = *reinterpret_cast<const uint4 *>(row + i);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const __half2 h = __floats2half2_rn(bf16_to_f32(w[q] & 0xFFFFu) * f, bf16_to_f32(w[q] >> 16) * f);
      o[q] = *reinterpret_cast<const uint32_t *>(&h);
    }
    *reinterpret_cast<uint4 *>(x16 + (size_t)t * H + i) = make_uint4(o[0], o[1], o[2], o[3]);
  }
  if (lane == 0) xshift[t] = sh;
}

// Decode routing: one CTA routes T <= 64 tokens (warp per token), builds the
// maps and the slot descriptors, and converts the activations for the GEMVs.
template <int N>
__global__ void __launch_bounds__(256) route_maps_fused_kernel(const float *__restrict__ logits, int T, int E,
                                                              int k, int normalize, RouteOut o) {
  extern __shared__ int32_t smem_i32[];
  pdl_launch_dependents();
  const int W = blockDim.x >> 5, w = (int)(threadIdx.x >> 5);
  for (int i = threadIdx.x; i < o.n_zero_words; i += blockDim.x) o.zero_words[i] = 0;
  for (int t = w; t < T; t += W) route_one_token<N>(logits, t, E, k, normalize, o.ids, o.weights);
  if (o.x) {
    for (int t = W - 1 - w; t < T; t += W) convert_token_fp16(o.x, o.H, t, o.x16, o.xshift);
  }
  __syncthreads();
  build_maps(o.ids, T * k, E, o.offsets, o.p2e, o.e2p, o.active, o.meta, o.slots, smem_i32, smem_i32 + W * E);
}

// Prefill routing, second step: one CTA of 1024 threads builds the maps.
__global__ void __launch_bounds__(1024) maps_kernel(int R, int E, RouteOut o) {
  extern __shared__ int32_t smem_i32[];
  const int W = blockDim.x >> 5;
  for (int i = threadIdx.x; i < o.n_zero_words; i += blockDim.x) o.zero_words[i] = 0;
  build_maps(o.ids, R, E, o.offsets, o.p2e, o.e2p, o.active, o.meta, o.slots, smem_i32, smem_i32 + W * E);
}

static int keys_per_lane(int E, int k) {
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
    const size_t smem = sizeof(int32_t) * ((size_t)W * E + E + 1);
    route_maps_fused_kernel<N><<<1, threads, smem, stream>>>(logits, T, E, k, normalize, o);
    return cudaGetLastError();
  }
  const int warps = 8;
  route_topk_kernel<N><<<(T + warps - 1) / warps, warps * 32, 0, stream>>>(logits, T, E, k, normalize, o.ids,
                                                                            o.weights);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  const int threads = 1024, W = threads / 32;
  const size_t smem = sizeof(int32_t) * ((size_t)W * E + E + 1);
  maps_kernel<<<1, threads, smem, stream>>>(T * k, E, o);
  return cudaGetLastError();
}

cudaError_t launch_route(const float *logits, int T, int E, int k, int normalize, const RouteOut &o,
                         cudaStream_t stream) {
  switch (keys_per_lane(E, k)) {
    case 1: return launch_route_n<1>(logits, T, E, k, normalize, o, stream);
    case 2: return launch_route_n<2>(logits, T, E, k, normalize, o, stream);
    case 4: return launch_route_n<4>(logits, T, E, k, normalize, o, stream);
    case 8: return launch_route_n<8>(logits, T, E, k, normalize, o, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace qmoe
