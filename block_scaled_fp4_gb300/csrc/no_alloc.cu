// qmoe_fp4_moe_forward_no_alloc: the MoE layer for callers that must not
// allocate device memory.
//
// Some callers cannot hand the layer a workspace: a plug-in that runs inside
// another engine's memory pool and is only given its input and output
// buffers, or a latency-critical loop where a cudaMalloc (which can stall the
// whole device) is not allowed once the loop is running.  This entry point
// serves them with scratch memory that lives in the library itself: a
// file-scope device array of kStaticScratchBytes, present on every GPU that
// loads the library until the process exits.  It forwards to
// qmoe_fp4_moe_forward, so the kernels, results and argument rules are
// exactly those of that call; it calls no cudaMalloc, cudaFree or allocating
// routine.
#include <mutex>

#include "qmoe_common.cuh"

namespace {

constexpr size_t kStaticScratchBytes = QMOE_NO_ALLOC_SCRATCH_BYTES;

// The scratch array.  In host code this name is only a host-side stand-in:
// the device address comes from cudaGetSymbolAddress, looked up once per
// device below.
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

std::mutex g_scratch_mutex;
void *g_scratch_addr[qmoe::kMaxDevices] = {nullptr};

}  // namespace

namespace qmoe {

// Device address of the scratch array on the current device (looked up on the
// first call for that device).
qmoe_status no_alloc_scratch(void **addr) {
  int dev = -1;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) {
    qmoe::set_error("no-alloc forward: cudaGetDevice failed: %s", cudaGetErrorString(err));
    return QMOE_ERR_CUDA;
  }
  if (dev < 0 || dev >= qmoe::kMaxDevices) {
    qmoe::set_error("no-alloc forward: device %d outside the supported range 0..%d", dev, qmoe::kMaxDevices - 1);
    return QMOE_ERR_UNSUPPORTED;
  }
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_addr[dev] == nullptr) {
    void *p = nullptr;
    err = cudaGetSymbolAddress(&p, g_static_scratch);
    if (err != cudaSuccess || p == nullptr) {
      qmoe::set_error("no-alloc forward: cudaGetSymbolAddress of the static scratch failed on device %d: %s", dev,
                      cudaGetErrorString(err));
      return QMOE_ERR_CUDA;
    }
    g_scratch_addr[dev] = p;
  }
  *addr = g_scratch_addr[dev];
  return QMOE_OK;
}

}  // namespace qmoe

extern "C" qmoe_status qmoe_fp4_moe_forward_no_alloc(const uint16_t *x, const float *logits, const uint8_t *fc1_w,
                                                     const uint8_t *fc1_s, const float *fc1_g,
                                                     const uint8_t *fc2_w, const uint8_t *fc2_s,
                                                     const float *fc2_g, qmoe_fp4_format fmt, int T, int H, int I,
                                                     int E, int k, int normalize, int swiglu_fusion, float alpha,
                                                     float beta, float limit, uint16_t *out,
                                                     int32_t *topk_ids_out, cudaStream_t stream) {
  // How much scratch this call needs (validates the sizes, launches nothing).
  size_t need = 0;
  qmoe_status st = qmoe_fp4_moe_forward(x, logits, nullptr, fc1_w, fc1_s, fc1_g, fc2_w, fc2_s, fc2_g, nullptr, nullptr, fmt,
                                        T, H, I, E, k, normalize, swiglu_fusion, alpha, beta, limit, out,
                                        topk_ids_out, nullptr, &need, stream);
  if (st != QMOE_OK) return st;
  if (need > kStaticScratchBytes) {
    qmoe::set_error("no-alloc forward: these sizes need %zu bytes of scratch but the library's static scratch "
                    "holds %zu bytes; use qmoe_fp4_moe_forward with a workspace",
                    need, kStaticScratchBytes);
    return QMOE_ERR_WORKSPACE;
  }
  void *scratch = nullptr;
  st = qmoe::no_alloc_scratch(&scratch);
  if (st != QMOE_OK) return st;
  size_t have = kStaticScratchBytes;
  // The array is zero when the module loads and its header stays zero between
  // calls (decode kernels leave it so; the prefill path never writes it).
  const qmoe_fp4_format primed = (qmoe_fp4_format)((int)fmt | (int)QMOE_WORKSPACE_PRIMED);
  return qmoe_fp4_moe_forward(x, logits, nullptr, fc1_w, fc1_s, fc1_g, fc2_w, fc2_s, fc2_g, nullptr, nullptr, primed, T, H,
                              I, E, k, normalize, swiglu_fusion, alpha, beta, limit, out, topk_ids_out, scratch,
                              &have, stream);
}
