// Router projection on the GPU: logits[t][e] = W_r[e] . x[t] for T <= 16
// tokens, W_r bf16 [E][H].
//
// flash-moe write-up (discuss.pytorch.kr), section "per-layer pipeline": the
// second command buffer computes the routing logits on the GPU before the
// softmax + top-K.  The projection reads E*H*2 bytes once (4 MiB for E 512,
// H 4096) and is bound by HBM latency at this size: each router row is read
// by four warps (a quarter of H each), two rows per block, so that E = 512
// spreads over 256 blocks; a lane issues all its 16-byte streaming loads of
// the row before any arithmetic (up to 8 in flight), and every loaded row
// chunk meets all T tokens from registers.  The sums are taken in a fixed
// order (lane, shuffle tree, then the four quarters), so the logits do not
// depend on scheduling.
#include "fmoe_kernels.cuh"

namespace fmoe {

namespace {

constexpr int kRtRowsPerBlock = 2;
constexpr int kRtWarpsPerRow = 4;
constexpr int kRtChunks = FMOE_MAX_HIDDEN / 8 / kRtWarpsPerRow / 32;   // 16-byte loads per lane, at most
constexpr int kRtThreads = 32 * kRtRowsPerBlock * kRtWarpsPerRow;

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__global__ void __launch_bounds__(kRtThreads) router_kernel(const uint16_t* __restrict__ w, const float* __restrict__ x,
                                                          int T, int H, int E, float* __restrict__ logits) {
  __shared__ float s_part[kRtRowsPerBlock][kRtWarpsPerRow][FMOE_MAX_TOKENS];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rl = warp / kRtWarpsPerRow, part = warp % kRtWarpsPerRow;
  const int row = blockIdx.x * kRtRowsPerBlock + rl;
  float acc[FMOE_MAX_TOKENS];
#pragma unroll
  for (int t = 0; t < FMOE_MAX_TOKENS; ++t) acc[t] = 0.f;
  if (row < E) {
    const int n8 = H / 8;                                   // 16-byte chunks of a row
    const int c0 = n8 * part / kRtWarpsPerRow, c1 = n8 * (part + 1) / kRtWarpsPerRow;
    const uint4* wr = reinterpret_cast<const uint4*>(w + (size_t)row * H);
    const float4* x4 = reinterpret_cast<const float4*>(x);
    uint4 q[kRtChunks];
#pragma unroll
    for (int j = 0; j < kRtChunks; ++j) {
      const int c = c0 + lane + 32 * j;
      q[j] = c < c1 ? ld_stream(wr + c) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int j = 0; j < kRtChunks; ++j) {
      const int c = c0 + lane + 32 * j;
      if (c < c1) {
        const float w0 = bf16lo(q[j].x), w1 = bf16hi(q[j].x), w2 = bf16lo(q[j].y), w3 = bf16hi(q[j].y);
        const float w4 = bf16lo(q[j].z), w5 = bf16hi(q[j].z), w6 = bf16lo(q[j].w), w7 = bf16hi(q[j].w);
#pragma unroll
        for (int t = 0; t < FMOE_MAX_TOKENS; ++t) {
          if (t < T) {
            const float4 a = __ldg(x4 + ((size_t)t * H >> 2) + 2 * c);
            const float4 b = __ldg(x4 + ((size_t)t * H >> 2) + 2 * c + 1);
            float s = acc[t];
            s = fmaf(w0, a.x, s);
            s = fmaf(w1, a.y, s);
            s = fmaf(w2, a.z, s);
            s = fmaf(w3, a.w, s);
            s = fmaf(w4, b.x, s);
            s = fmaf(w5, b.y, s);
            s = fmaf(w6, b.z, s);
            s = fmaf(w7, b.w, s);
            acc[t] = s;
          }
        }
      }
    }
  }
#pragma unroll
  for (int t = 0; t < FMOE_MAX_TOKENS; ++t) {
    if (t < T) {
      const float v = warp_sum(acc[t]);
      if (lane == 0) s_part[rl][part][t] = v;
    }
  }
  __syncthreads();
  const int i = threadIdx.x;
  if (i < kRtRowsPerBlock * T) {
    const int r = i / T, t = i - r * T;
    const int e = blockIdx.x * kRtRowsPerBlock + r;
    if (e < E) {
      float v = 0.f;
#pragma unroll
      for (int h2 = 0; h2 < kRtWarpsPerRow; ++h2) v += s_part[r][h2][t];
      logits[(size_t)t * E + e] = v;
    }
  }
}

}  // namespace

cudaError_t launch_router(const uint16_t* w, const float* x, int T, int H, int E, float* logits, cudaStream_t st) {
  const int blocks = (E + kRtRowsPerBlock - 1) / kRtRowsPerBlock;
  router_kernel<<<blocks, kRtThreads, 0, st>>>(w, x, T, H, E, logits);
  return cudaGetLastError();
}

}  // namespace fmoe
