// fmoe_moe_block_noalloc: the single-token MoE block for callers that cannot
// allocate device memory.
//
// Some callers have no way to hand the library a workspace: code that runs
// where cudaMalloc is not allowed or not wanted (inside a custom allocator or
// memory-pool callback, in a plugin whose host framework owns every device
// allocation, or in a hard-real-time loop where an allocation may block).
// For them this file keeps the scratch the single-launch kernel needs (error
// word, exit counter, layer count and the fixed-point accumulators through
// which its blocks add up their partial outputs) in one file-scope
// __device__ array.  That array is part of the
// library image: every GPU that loads libfmoe.so holds its
// FMOE_NOALLOC_SCRATCH_BYTES bytes until the process exits.
//
// Host code cannot use the array's name as a device address (on the host it
// names a host-side shadow), so every call asks the runtime for the array's
// device address on the current device with cudaGetSymbolAddress.  Once the
// library's device code is loaded on a device this is a host-side lookup; the
// first call on a device loads it, which is why that first call should come
// before any stream capture.  Looking the address up each time (rather than
// caching it per device) keeps it right after cudaDeviceReset or under
// another context, where the array may be reloaded at a different address.
#include "fmoe_kernels.cuh"

using namespace fmoe;

namespace {

static_assert(FMOE_NOALLOC_SCRATCH_BYTES % 256 == 0, "scratch size must be a multiple of 256");

__device__ __align__(256) uint8_t g_noalloc_scratch[FMOE_NOALLOC_SCRATCH_BYTES];

constexpr unsigned long long kNoallocTimeoutNs = 200ull * 1000 * 1000;

// Device address of the scratch array on the current device; nullptr on failure.
void* scratch_on_current_device() {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return p;
}

}  // namespace

extern "C" fmoe_status fmoe_moe_block_noalloc(const fmoe_layer* layer, const float* x,
                                              const float* router_logits, const float* residual,
                                              float* out, int K, uint32_t* device_error, void* stream) {
  fmoe_status s = check_layer(layer, true);
  if (s != FMOE_OK) return s;
  if (K < 1 || K > FMOE_MAX_TOPK || K > layer->n_experts) return FMOE_ERR_INVALID_ARG;
  s = check_block_args(layer, x, router_logits, residual, out, 1);
  if (s != FMOE_OK) return s;
  if (device_error != nullptr && !host_aligned(device_error, 4)) return FMOE_ERR_INVALID_ARG;

  // The kernel's scratch: the header (error word, exit count, layer count)
  // and its three accumulators, 256 + 24*H bytes rounded up to 256 (98,560
  // bytes at H = 4096); larger hidden sizes are refused.
  const int S = layer->has_shared;
  const WsLayout wl = ws_layout(layer->hidden, layer->inter, S, 1, K, 1);
  if (wl.state > (size_t)FMOE_NOALLOC_SCRATCH_BYTES) return FMOE_ERR_INVALID_ARG;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return FMOE_ERR_CUDA;
  }
  const FusedPlan pl = fused_plan(layer->bits, layer->hidden, layer->inter, K, S, dev);
  if (!pl.ok) return FMOE_ERR_UNSUPPORTED;
  uint8_t* base = static_cast<uint8_t*>(scratch_on_current_device());
  if (base == nullptr) return FMOE_ERR_CUDA;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // Every call starts from a clean state: the error word, the exit count,
  // the layer count and the accumulators (the previous call, or one that
  // timed out, may have left them otherwise).
  cudaError_t e = cudaMemsetAsync(base, 0, wl.state, st);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return FMOE_ERR_CUDA;
  }

  FusedParams p{};
  fused_params_for(p, layer, 1, K);
  p.norm = 0;
  p.eps = 0.f;
  p.x = x;
  p.residual = residual;
  p.out = out;
  p.logits = router_logits;
  p.hmid = nullptr;
  p.acc = reinterpret_cast<unsigned long long*>(base + wl.acc);
  p.lbase = reinterpret_cast<uint32_t*>(base + wl.lbase);
  p.ids_out = nullptr;
  p.w_out = nullptr;
  p.gate_out = nullptr;
  p.exit_ctr = reinterpret_cast<uint32_t*>(base + wl.exit_ctr);
  p.err = reinterpret_cast<uint32_t*>(base + wl.err);
  p.timeout_ns = kNoallocTimeoutNs;
  e = launch_fused(p, pl, st);
  if (e == cudaSuccess && device_error != nullptr)
    e = cudaMemcpyAsync(device_error, base + wl.err, sizeof(uint32_t), cudaMemcpyDeviceToDevice, st);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return FMOE_ERR_CUDA;
  }
  return FMOE_OK;
}
