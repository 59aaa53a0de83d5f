// fmoe_moe_block_noalloc: the single-token MoE block for callers that cannot
// allocate device memory.
//
// Some callers have no way to hand the library a workspace: code that runs
// where cudaMalloc is not allowed or not wanted (inside a custom allocator or
// memory-pool callback, in a plugin whose host framework owns every device
// allocation, or in a hard-real-time loop where an allocation may block).
// For them this file keeps the scratch the single-launch kernel needs
// (error word, exit counter, launch epoch, routing result, intermediate
// activations) in one file-scope __device__ array.  That array is part of the
// library image: every GPU that loads libfmoe.so holds its
// FMOE_NOALLOC_SCRATCH_BYTES bytes until the process exits.
//
// Host code cannot use the array's name as a device address (on the host it
// names a host-side shadow), so the device address is looked up once per
// device with cudaGetSymbolAddress, with that device current, and cached.
#include <mutex>

#include "fmoe_kernels.cuh"

using namespace fmoe;

namespace {

static_assert(FMOE_NOALLOC_SCRATCH_BYTES % 256 == 0, "scratch size must be a multiple of 256");

__device__ __align__(256) uint8_t g_noalloc_scratch[FMOE_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
constexpr unsigned long long kNoallocTimeoutNs = 200ull * 1000 * 1000;

std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up on
// the first call per device).  nullptr on failure.
void* scratch_on_current_device(int dev) {
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    g_scratch_addr[dev] = p;
  }
  return g_scratch_addr[dev];
}

bool is_aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const char* pa = static_cast<const char*>(a);
  const char* pb = static_cast<const char*>(b);
  return pa < pb + nb && pb < pa + na;
}

}  // namespace

extern "C" fmoe_status fmoe_moe_block_noalloc(const fmoe_layer* layer, const float* x,
                                              const float* router_logits, const float* residual,
                                              float* out, int K, uint32_t* device_error, void* stream) {
  if (layer == nullptr) return FMOE_ERR_INVALID_ARG;
  if (layer->bits != 4 && layer->bits != 2) return FMOE_ERR_UNSUPPORTED;
  if (layer->group != kGroup) return FMOE_ERR_UNSUPPORTED;
  if (layer->hidden <= 0 || layer->inter <= 0 || layer->hidden % kGroup || layer->inter % kGroup)
    return FMOE_ERR_INVALID_ARG;
  if (layer->hidden > FMOE_MAX_HIDDEN || layer->inter > FMOE_MAX_INTER) return FMOE_ERR_UNSUPPORTED;
  if (layer->n_experts <= 0 || layer->n_experts > FMOE_MAX_EXPERTS) return FMOE_ERR_INVALID_ARG;
  if (layer->has_shared != 0 && layer->has_shared != 1) return FMOE_ERR_INVALID_ARG;
  if (layer->experts == nullptr || !is_aligned(layer->experts, kPlaneAlign)) return FMOE_ERR_INVALID_ARG;
  if (layer->has_shared &&
      (layer->shared == nullptr || !is_aligned(layer->shared, kPlaneAlign) || layer->shared_gate_w == nullptr ||
       !is_aligned(layer->shared_gate_w, 16)))
    return FMOE_ERR_INVALID_ARG;
  if (K < 1 || K > FMOE_MAX_TOPK || K > layer->n_experts) return FMOE_ERR_INVALID_ARG;
  for (const void* p : {static_cast<const void*>(x), static_cast<const void*>(router_logits),
                        static_cast<const void*>(residual), static_cast<const void*>(out)})
    if (p == nullptr || !is_aligned(p, 16)) return FMOE_ERR_INVALID_ARG;
  if (device_error != nullptr && !is_aligned(device_error, 4)) return FMOE_ERR_INVALID_ARG;
  const size_t hb = (size_t)layer->hidden * 4;
  if (overlaps(out, hb, x, hb) || overlaps(out, hb, router_logits, (size_t)layer->n_experts * 4))
    return FMOE_ERR_INVALID_ARG;
  if (out != residual && overlaps(out, hb, residual, hb)) return FMOE_ERR_INVALID_ARG;

  const int S = layer->has_shared;
  const WsLayout wl = ws_layout(layer->hidden, layer->inter, S, 1, K, 1);
  if (wl.bytes > (size_t)FMOE_NOALLOC_SCRATCH_BYTES) return FMOE_ERR_INVALID_ARG;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return FMOE_ERR_CUDA;
  }
  const FusedPlan pl = fused_plan(layer->bits, layer->hidden, layer->inter, K, S, dev);
  if (!pl.ok) return FMOE_ERR_UNSUPPORTED;
  uint8_t* base = static_cast<uint8_t*>(scratch_on_current_device(dev));
  if (base == nullptr) return FMOE_ERR_CUDA;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // The error word and the count of finished blocks must start at zero; the
  // previous call (or a timed-out one) may have left them otherwise.  The
  // launch counter that tags the blocks' exchanges must never go back, so it
  // is left alone.
  cudaError_t e = cudaMemsetAsync(base, 0, wl.header_clear, st);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return FMOE_ERR_CUDA;
  }

  FusedParams p{};
  p.bits = layer->bits;
  p.H = layer->hidden;
  p.I = layer->inter;
  p.E = layer->n_experts;
  p.K = K;
  p.S = S;
  p.L = 1;
  p.norm = 0;
  p.eps = 0.f;
  p.lay = blob_layout(layer->bits, layer->hidden, layer->inter);
  p.blob = p.lay.bytes;
  p.x = x;
  p.residual = residual;
  p.out = out;
  p.logits = router_logits;
  p.hmid = reinterpret_cast<float*>(base + wl.h);
  p.hll = reinterpret_cast<unsigned long long*>(base + wl.hll);
  p.hbufll = reinterpret_cast<unsigned long long*>(base + wl.hbufll);
  p.ids_out = nullptr;
  p.w_out = nullptr;
  p.gate_out = nullptr;
  p.exit_ctr = reinterpret_cast<uint32_t*>(base + wl.exit_ctr);
  p.epoch = reinterpret_cast<uint32_t*>(base + wl.epoch);
  p.err = reinterpret_cast<uint32_t*>(base + wl.err);
  p.timeout_ns = kNoallocTimeoutNs;
  p.layer[0].experts = static_cast<const uint8_t*>(layer->experts);
  p.layer[0].shared = static_cast<const uint8_t*>(layer->shared);
  p.layer[0].wsg = layer->shared_gate_w;
  e = launch_fused(p, pl, st);
  if (e == cudaSuccess && device_error != nullptr)
    e = cudaMemcpyAsync(device_error, base + wl.err, sizeof(uint32_t), cudaMemcpyDeviceToDevice, st);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return FMOE_ERR_CUDA;
  }
  return FMOE_OK;
}
