// Routing kernel and the general (any T, any supported shape) expert kernels.
//
// These kernels give every entry point a CUDA path for every shape the ABI
// accepts; the single-launch persistent kernel (fmoe_fused.cu) is the fast
// path for batch-1 blocks and stacks, the batched kernels (fmoe_batch.cu)
// the fast path for T > 1.
//
// Sources: flash-moe write-up (discuss.pytorch.kr): "per-layer pipeline"
// (softmax + top-K routing, expert forward, combine), "hand-written Metal
// compute shaders" (dequant matvec, fused SwiGLU, MoE combine + residual +
// sigmoid gate), "FMA-optimised dequant kernel" (code * scale + bias).
#include "fmoe_kernels.cuh"

namespace fmoe {

// One warp per token: top-K + softmax, and the shared-expert gate
// g = sigmoid(w_sg . x) when wsg != nullptr.
__global__ void route_kernel(const float* __restrict__ logits, int T, int E, int K,
                             int32_t* __restrict__ ids, float* __restrict__ weights,
                             const uint16_t* __restrict__ wsg, const float* __restrict__ x, int H,
                             float* __restrict__ gate) {
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  int id; float w;
  warp_route(logits + (size_t)t * E, E, K, id, w);
  if (lane < K) {
    ids[(size_t)t * K + lane] = id;
    weights[(size_t)t * K + lane] = w;
  }
  if (gate != nullptr) {
    float acc = 0.f;
    if (wsg != nullptr) {
      for (int c = lane; c < H; c += 32) acc += bf16v(wsg[c]) * x[(size_t)t * H + c];
      acc = warp_sum(acc);
    }
    if (lane == 0) gate[t] = (wsg != nullptr) ? sigmoid_f(acc) : 0.f;
  }
}

__device__ __forceinline__ const uint8_t* slot_blob(const GenericArgs& a, int t, int slot) {
  if (slot < a.K) {
    const int id = a.ids[(size_t)t * a.K + slot];
    if (id < 0 || id >= a.E) {
      atomicOr(a.err, kErrBadExpert);
      return nullptr;
    }
    return a.experts + (size_t)id * a.blob;
  }
  return a.shared;
}

template <int BITS>
__device__ __forceinline__ SliceCodes<BITS> load_codes(const uint8_t* row, int s) {
  SliceCodes<BITS> q;
  if constexpr (BITS == 4) q.v = __ldg(reinterpret_cast<const uint4*>(row) + s);
  else q.v = __ldg(reinterpret_cast<const uint2*>(row) + s);
  return q;
}

// One warp per (token t, slot, intermediate row r):
//   h[t][slot][r] = silu(gate_r . x_t) * (up_r . x_t)
template <int BITS>
__global__ void gateup_generic_kernel(GenericArgs a) {
  const long long gw = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const int NS = a.K + a.S;
  const long long total = (long long)a.T * NS * a.I;
  if (gw >= total) return;
  const int r = (int)(gw % a.I);
  const int slot = (int)((gw / a.I) % NS);
  const int t = (int)(gw / ((long long)a.I * NS));
  const uint8_t* blob = slot_blob(a, t, slot);
  float* hout = a.h + ((size_t)t * NS + slot) * a.I + r;
  if (blob == nullptr) { if (lane == 0) *hout = 0.f; return; }
  const uint8_t* row = blob + (size_t)r * a.lay.gu_row;
  const uint8_t* gq = row;
  const uint8_t* uq = row + a.lay.qh;
  const uint32_t* gsb = reinterpret_cast<const uint32_t*>(row + 2 * a.lay.qh);
  const uint32_t* usb = reinterpret_cast<const uint32_t*>(row + 2 * a.lay.qh + a.lay.sh);
  const float* x = a.x + (size_t)t * a.H;
  float ga = 0.f, ua = 0.f;
  for (int s = lane; s < a.H / kSlice; s += 32) {
    SliceX xs;
    const float xsum = load_slice_x<BITS, false>(x, s, 1.0f, xs);
    ga += slice_term<BITS>(load_codes<BITS>(gq, s), __ldg(gsb + s / 2), xs, xsum);
    ua += slice_term<BITS>(load_codes<BITS>(uq, s), __ldg(usb + s / 2), xs, xsum);
  }
  ga = warp_sum(ga);
  ua = warp_sum(ua);
  if (lane == 0) *hout = silu_f(ga) * ua;
}

// One warp per (token t, slot, output row j): y[t][slot][j] = down_j . h[t][slot]
template <int BITS>
__global__ void down_y_kernel(GenericArgs a, float* __restrict__ y) {
  const long long gw = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const int NS = a.K + a.S;
  const long long total = (long long)a.T * NS * a.H;
  if (gw >= total) return;
  const int j = (int)(gw % a.H);
  const int slot = (int)((gw / a.H) % NS);
  const int t = (int)(gw / ((long long)a.H * NS));
  const uint8_t* blob = slot_blob(a, t, slot);
  float* yout = y + ((size_t)t * NS + slot) * a.H + j;
  if (blob == nullptr) { if (lane == 0) *yout = 0.f; return; }
  const uint8_t* dq = blob + a.lay.d_off + (size_t)j * a.lay.d_row;
  const uint32_t* dsb = reinterpret_cast<const uint32_t*>(dq + a.lay.qi);
  const float* h = a.h + ((size_t)t * NS + slot) * a.I;
  float acc = 0.f;
  for (int s = lane; s < a.I / kSlice; s += 32) {
    SliceX hs;
    const float hsum = load_slice_x<BITS, false>(h, s, 1.0f, hs);
    acc += slice_term<BITS>(load_codes<BITS>(dq, s), __ldg(dsb + s / 2), hs, hsum);
  }
  acc = warp_sum(acc);
  if (lane == 0) *yout = acc;
}

// One warp per (token t, output row j):
//   out[t][j] = residual[t][j] + sum_k w[t][k] y_k[j] + gate[t] y_shared[j]
template <int BITS>
__global__ void down_combine_kernel(GenericArgs a) {
  const long long gw = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const int NS = a.K + a.S;
  if (gw >= (long long)a.T * a.H) return;
  const int j = (int)(gw % a.H);
  const int t = (int)(gw / a.H);
  float acc = 0.f;
  for (int slot = 0; slot < NS; ++slot) {
    const uint8_t* blob = slot_blob(a, t, slot);
    if (blob == nullptr) continue;
    const float wk = (slot < a.K) ? a.weights[(size_t)t * a.K + slot] : a.gate[t];
    const uint8_t* dq = blob + a.lay.d_off + (size_t)j * a.lay.d_row;
    const uint32_t* dsb = reinterpret_cast<const uint32_t*>(dq + a.lay.qi);
    const float* h = a.h + ((size_t)t * NS + slot) * a.I;
    float part = 0.f;
    for (int s = lane; s < a.I / kSlice; s += 32) {
      SliceX hs;
      const float hsum = load_slice_x<BITS, false>(h, s, 1.0f, hs);
      part += slice_term<BITS>(load_codes<BITS>(dq, s), __ldg(dsb + s / 2), hs, hsum);
    }
    acc = fmaf(wk, part, acc);
  }
  acc = warp_sum(acc);
  if (lane == 0) a.out[(size_t)t * a.H + j] = a.residual[(size_t)t * a.H + j] + acc;
}

// ---------------------------------------------------------------------------
// host launchers
// ---------------------------------------------------------------------------
cudaError_t launch_route(const float* logits, int T, int E, int K, int32_t* ids, float* weights,
                         const uint16_t* wsg, const float* x, int H, float* gate, cudaStream_t st) {
  const int warps = 4;
  route_kernel<<<(T + warps - 1) / warps, 32 * warps, 0, st>>>(logits, T, E, K, ids, weights, wsg, x,
                                                                 H, gate);
  return cudaGetLastError();
}

static inline unsigned warp_blocks(long long warps, int per_block) {
  return (unsigned)((warps + per_block - 1) / per_block);
}

cudaError_t launch_gateup_generic(const GenericArgs& a, cudaStream_t st) {
  const long long warps = (long long)a.T * (a.K + a.S) * a.I;
  if (a.bits == 4) gateup_generic_kernel<4><<<warp_blocks(warps, 8), 256, 0, st>>>(a);
  else gateup_generic_kernel<2><<<warp_blocks(warps, 8), 256, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_down_y(const GenericArgs& a, float* y, cudaStream_t st) {
  const long long warps = (long long)a.T * (a.K + a.S) * a.H;
  if (a.bits == 4) down_y_kernel<4><<<warp_blocks(warps, 8), 256, 0, st>>>(a, y);
  else down_y_kernel<2><<<warp_blocks(warps, 8), 256, 0, st>>>(a, y);
  return cudaGetLastError();
}

cudaError_t launch_down_combine(const GenericArgs& a, cudaStream_t st) {
  const long long warps = (long long)a.T * a.H;
  if (a.bits == 4) down_combine_kernel<4><<<warp_blocks(warps, 8), 256, 0, st>>>(a);
  else down_combine_kernel<2><<<warp_blocks(warps, 8), 256, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace fmoe
