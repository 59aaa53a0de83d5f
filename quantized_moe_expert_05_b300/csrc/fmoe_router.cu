// Router projection on the GPU: logits[t][e] = W_r[e] . x[t] for T <= 16
// tokens, W_r bf16 [E][H].
//
// flash-moe write-up (discuss.pytorch.kr), section "per-layer pipeline": the
// second command buffer computes the routing logits on the GPU before the
// softmax + top-K.  The projection reads E*H*2 bytes once (4 MiB for E 512,
// H 4096).  Each group of RPW router rows is read by four warps (a quarter
// of H each), two groups per block; a lane issues its 16-byte streaming
// loads of a pass (all of them for one row, two chunks of every row for
// several) before any arithmetic, and every token's inputs, loaded once,
// meet all RPW rows from registers.  The sums are taken in a fixed order
// (lane, shuffle tree, then the four quarters), so the logits do not depend
// on scheduling.
#include "fmoe_kernels.cuh"

namespace fmoe {

namespace {

constexpr int kRtGroupsPerBlock = 2;
constexpr int kRtWarpsPerRow = 4;
constexpr int kRtChunks = FMOE_MAX_HIDDEN / 8 / kRtWarpsPerRow / 32;   // 16-byte loads per lane and row, at most
constexpr int kRtThreads = 32 * kRtGroupsPerBlock * kRtWarpsPerRow;
constexpr int kRtMaxRows = 4;                              // bound on rt_rows()

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// rows of a group, measured at E 512, H 4096 (8 projections in one graph,
// against a kernel holding 16 tokens always, one row per group): one row
// (256 blocks for E 512) takes T 1 from 6.5 to 3.3 us, T 4 from 8.5 to 6.2
// and T 16 from 17.2 to 16.2; at two tokens, two rows (128 blocks) sharing
// each input load take 5.5 us against 7.4.  Two rows from four tokens on
// ran slower (T 16: 21.2 us), four rows (64 blocks) slower still (25.4).
__host__ __device__ constexpr int rt_rows(int NT) { return NT == 2 ? 2 : 1; }

// NT: tokens held in registers, the smallest of 1, 2, 4, 8, 16 that is >= T.
template <int NT>
__global__ void __launch_bounds__(kRtThreads, 1) router_kernel(const uint16_t* __restrict__ w, const float* __restrict__ x,
                                                          int T, int H, int E, float* __restrict__ logits) {
  constexpr int RPW = rt_rows(NT);
  constexpr int PASS = RPW == 1 ? kRtChunks : 2;          // chunks per lane and row loaded before their arithmetic
  __shared__ float s_part[kRtGroupsPerBlock][kRtWarpsPerRow][kRtMaxRows][NT];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rg = warp / kRtWarpsPerRow, part = warp % kRtWarpsPerRow;
  const int row0 = (blockIdx.x * kRtGroupsPerBlock + rg) * RPW;
  float acc[RPW][NT];
#pragma unroll
  for (int r = 0; r < RPW; ++r)
#pragma unroll
    for (int t = 0; t < NT; ++t) acc[r][t] = 0.f;
  if (row0 < E) {
    const int n8 = H / 8;                                   // 16-byte chunks of a row
    const int c0 = n8 * part / kRtWarpsPerRow, c1 = n8 * (part + 1) / kRtWarpsPerRow;
    const uint4* wr[RPW];
#pragma unroll
    for (int r = 0; r < RPW; ++r)   // a row past the last is read as the last again; its sums are dropped
      wr[r] = reinterpret_cast<const uint4*>(w + (size_t)min(row0 + r, E - 1) * H);
    const float4* x4 = reinterpret_cast<const float4*>(x);
#pragma unroll
    for (int j0 = 0; j0 < kRtChunks; j0 += PASS) {
      uint4 q[PASS][RPW];
#pragma unroll
      for (int j = 0; j < PASS; ++j) {
        const int c = c0 + lane + 32 * (j0 + j);
#pragma unroll
        for (int r = 0; r < RPW; ++r) q[j][r] = c < c1 ? ld_stream(wr[r] + c) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int j = 0; j < PASS; ++j) {
        const int c = c0 + lane + 32 * (j0 + j);
        if (c < c1) {
          float wv[RPW][8];
#pragma unroll
          for (int r = 0; r < RPW; ++r) {
            wv[r][0] = bf16lo(q[j][r].x);
            wv[r][1] = bf16hi(q[j][r].x);
            wv[r][2] = bf16lo(q[j][r].y);
            wv[r][3] = bf16hi(q[j][r].y);
            wv[r][4] = bf16lo(q[j][r].z);
            wv[r][5] = bf16hi(q[j][r].z);
            wv[r][6] = bf16lo(q[j][r].w);
            wv[r][7] = bf16hi(q[j][r].w);
          }
#pragma unroll
          for (int t = 0; t < NT; ++t) {
            if (t < T) {
              const float4 a = __ldg(x4 + ((size_t)t * H >> 2) + 2 * c);
              const float4 b = __ldg(x4 + ((size_t)t * H >> 2) + 2 * c + 1);
#pragma unroll
              for (int r = 0; r < RPW; ++r) {
                float v = acc[r][t];
                v = fmaf(wv[r][0], a.x, v);
                v = fmaf(wv[r][1], a.y, v);
                v = fmaf(wv[r][2], a.z, v);
                v = fmaf(wv[r][3], a.w, v);
                v = fmaf(wv[r][4], b.x, v);
                v = fmaf(wv[r][5], b.y, v);
                v = fmaf(wv[r][6], b.z, v);
                v = fmaf(wv[r][7], b.w, v);
                acc[r][t] = v;
              }
            }
          }
        }
      }
    }
  }
#pragma unroll
  for (int r = 0; r < RPW; ++r) {
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      if (t < T) {
        const float v = warp_sum(acc[r][t]);
        if (lane == 0) s_part[rg][part][r][t] = v;
      }
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < kRtGroupsPerBlock * RPW * T; i += kRtThreads) {
    const int t = i % T, rr = i / T;
    const int g = rr / RPW, r = rr % RPW;
    const int e = (blockIdx.x * kRtGroupsPerBlock + g) * RPW + r;
    if (e < E) {
      float v = 0.f;
#pragma unroll
      for (int h2 = 0; h2 < kRtWarpsPerRow; ++h2) v += s_part[g][h2][r][t];
      logits[(size_t)t * E + e] = v;
    }
  }
}

}  // namespace

cudaError_t launch_router(const uint16_t* w, const float* x, int T, int H, int E, float* logits, cudaStream_t st) {
#define FMOE_RT(NT)                                                                                  \
  router_kernel<NT><<<(E + kRtGroupsPerBlock * rt_rows(NT) - 1) / (kRtGroupsPerBlock * rt_rows(NT)), kRtThreads, 0, \
                      st>>>(w, x, T, H, E, logits)
  if (T <= 1) FMOE_RT(1);
  else if (T <= 2) FMOE_RT(2);
  else if (T <= 4) FMOE_RT(4);
  else if (T <= 8) FMOE_RT(8);
  else FMOE_RT(16);
#undef FMOE_RT
  return cudaGetLastError();
}

}  // namespace fmoe
