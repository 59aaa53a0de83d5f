// The MoE-adjacent steps of a layer: the dense quantised matrix-vector
// product of the attention output projection (o_proj), with the residual
// added, and RMSNorm with a learned weight.
//
// flash-moe write-up (discuss.pytorch.kr), section "per-layer pipeline": the
// second command buffer runs o_proj, the norm, the routing logits and the
// shared expert on the GPU; section "hand-written Metal compute shaders": a
// two-stage RMS normalisation and the 4-bit dequant matvec.
//
// A dense matrix is N row records (the row's codes, then one (scale,bias)
// word per 64 columns, padded to 16 bytes).  One warp computes RPW (1, 2 or
// 4) output rows for all T <= 16 tokens (the kernel is instantiated for 1,
// 2, 4, 8 and 16 tokens held in registers): lane l takes code word l of
// every 128-byte span of its rows (coalesced loads of codes and of the
// inputs they meet), issues several words of every row before their
// arithmetic, unpacks each word once, and meets each token's inputs, loaded
// once, with all RPW rows, adding s * sum(q * x) + b * sum(x) with the
// word's group scale and bias.  Sums are taken in a fixed order (words in
// order within a lane, then a shuffle tree), so results are deterministic.
#include "fmoe_kernels.cuh"

namespace fmoe {

namespace {

constexpr int kDgWarps = 4;
constexpr int kDgThreads = 32 * kDgWarps;

__device__ __forceinline__ uint32_t ld_stream_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

// rows per warp, measured at H 4096 (8 o_proj launches in one graph):
// 4-bit, one row for one or two tokens (T 2: 12.0 us against 13.9 with two
// rows; T 1 the same, 8.5 us) and four rows from four tokens on, where every
// input load serves four rows (T 16: 88 us against 112 with one row); 2-bit,
// two rows throughout (T 1: 8.2 against 11.4 us; T 16: 76 against 144 us).
// Loading sixteen words per row before the arithmetic at T 1 instead of
// eight was slower (8.7 and 9.0 us).
template <int BITS, int NT>
__host__ __device__ constexpr int dg_rows() {
  return BITS == 4 ? (NT <= 2 ? 1 : 4) : 2;
}

// NT: tokens held in registers, the smallest of 1, 2, 4, 8, 16 that is >= T.
template <int BITS, int NT>
__global__ void __launch_bounds__(kDgThreads) dense_gemv_kernel(const uint8_t* __restrict__ w, int N, int H, int rec,
                                                              const float* __restrict__ x, int T,
                                                              const float* residual, float* y) {
  constexpr int CPW = 32 / BITS;                        // columns per 32-bit word
  constexpr int RPW = dg_rows<BITS, NT>();              // rows per warp
  constexpr int PASS = NT >= 4 ? 4 : 8;                 // words per lane and row loaded before their arithmetic
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row0 = (blockIdx.x * kDgWarps + warp) * RPW;
  if (row0 >= N) return;                                // whole warps only: no barrier below
  const uint32_t* codes[RPW];
  const uint32_t* sbw[RPW];
#pragma unroll
  for (int r = 0; r < RPW; ++r) {
    // a row past the last is read as the last row again; its sums are dropped
    const uint8_t* rp = w + (size_t)min(row0 + r, N - 1) * rec;
    codes[r] = reinterpret_cast<const uint32_t*>(rp);
    sbw[r] = reinterpret_cast<const uint32_t*>(rp + (size_t)H * BITS / 8);
  }
  const int nwt = H / CPW;                              // code words of a row (H is a multiple of 64)
  const int nw = (nwt + 31) / 32;                       // rounds of 32 words
  float acc[RPW][NT];
#pragma unroll
  for (int r = 0; r < RPW; ++r)
#pragma unroll
    for (int t = 0; t < NT; ++t) acc[r][t] = 0.f;
  for (int p0 = 0; p0 < nw; p0 += PASS) {
    uint32_t q[PASS][RPW];
#pragma unroll
    for (int j = 0; j < PASS; ++j)
#pragma unroll
      for (int r = 0; r < RPW; ++r) {
        const int wi = 32 * (p0 + j) + lane;
        q[j][r] = wi < nwt ? ld_stream_u32(codes[r] + wi) : 0u;
      }
#pragma unroll
    for (int j = 0; j < PASS; ++j) {
      if (32 * (p0 + j) + lane < nwt) {
        const int c0 = (32 * (p0 + j) + lane) * CPW;     // the word's first column
        float s[RPW], b[RPW], qv[RPW][CPW];
#pragma unroll
        for (int r = 0; r < RPW; ++r) {
          const uint32_t sb = __ldg(sbw[r] + c0 / kGroup);
          s[r] = bf16lo(sb);
          b[r] = bf16hi(sb);
#pragma unroll
          for (int i = 0; i < CPW; ++i) qv[r][i] = (float)((q[j][r] >> (BITS * i)) & ((1u << BITS) - 1u));
        }
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          if (t < T) {
            const float4* xp = reinterpret_cast<const float4*>(x + (size_t)t * H + c0);
            float xv[CPW];
#pragma unroll
            for (int v = 0; v < CPW / 4; ++v) {
              const float4 a = __ldg(xp + v);
              xv[4 * v] = a.x;
              xv[4 * v + 1] = a.y;
              xv[4 * v + 2] = a.z;
              xv[4 * v + 3] = a.w;
            }
            float sx = 0.f;
#pragma unroll
            for (int v = 0; v < CPW / 4; ++v) sx += (xv[4 * v] + xv[4 * v + 1]) + (xv[4 * v + 2] + xv[4 * v + 3]);
#pragma unroll
            for (int r = 0; r < RPW; ++r) {
              float sq = 0.f;
#pragma unroll
              for (int i = 0; i < CPW; ++i) sq = fmaf(qv[r][i], xv[i], sq);
              acc[r][t] = fmaf(s[r], sq, fmaf(b[r], sx, acc[r][t]));
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
        const int row = row0 + r;
        if (lane == 0 && row < N) {
          const size_t o = (size_t)t * N + row;
          y[o] = residual != nullptr ? residual[o] + v : v;
        }
      }
    }
  }
}

// One block per token: x = h / sqrt(mean(h^2) + eps) (* w when given); the
// sum of squares in a fixed order (strided per thread, shuffle tree per
// warp, warps in order).  x may be h.
__global__ void __launch_bounds__(kNormThreads) rmsnorm_w_kernel(const float* h, const float* __restrict__ w, int H,
                                                                float eps, float* x) {
  __shared__ float s_part[kNormThreads / 32];
  __shared__ float s_rinv;
  const float* ht = h + (size_t)blockIdx.x * H;
  float* xt = x + (size_t)blockIdx.x * H;
  float ss = 0.f;
  for (int j = threadIdx.x; j < H; j += kNormThreads) {
    const float v = __ldcg(ht + j);
    ss += v * v;
  }
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) s_part[threadIdx.x >> 5] = ss;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.f;
    for (int k = 0; k < kNormThreads / 32; ++k) t += s_part[k];
    s_rinv = 1.0f / sqrtf(t / (float)H + eps);
  }
  __syncthreads();
  for (int j = threadIdx.x; j < H; j += kNormThreads) {
    const float v = __ldcg(ht + j) * s_rinv;
    xt[j] = w != nullptr ? v * __ldg(w + j) : v;
  }
}

}  // namespace

int dense_row_bytes(int bits, int H) {
  const int qb = H * bits / 8, sb = H / kGroup * 4;
  return (qb + sb + 15) / 16 * 16;
}

cudaError_t launch_dense_gemv(const uint8_t* w, int bits, int N, int H, const float* x, int T, const float* residual,
                              float* y, cudaStream_t st) {
  const int rec = dense_row_bytes(bits, H);
#define FMOE_DG(B, NT)                                                                      \
  dense_gemv_kernel<B, NT><<<(N + kDgWarps * dg_rows<B, NT>() - 1) / (kDgWarps * dg_rows<B, NT>()), kDgThreads, 0, \
                             st>>>(w, N, H, rec, x, T, residual, y)
  if (bits == 4) {
    if (T <= 1) FMOE_DG(4, 1);
    else if (T <= 2) FMOE_DG(4, 2);
    else if (T <= 4) FMOE_DG(4, 4);
    else if (T <= 8) FMOE_DG(4, 8);
    else FMOE_DG(4, 16);
  } else {
    if (T <= 1) FMOE_DG(2, 1);
    else if (T <= 2) FMOE_DG(2, 2);
    else if (T <= 4) FMOE_DG(2, 4);
    else if (T <= 8) FMOE_DG(2, 8);
    else FMOE_DG(2, 16);
  }
#undef FMOE_DG
  return cudaGetLastError();
}

cudaError_t launch_rmsnorm_w(const float* h, const float* w, int T, int H, float eps, float* x, cudaStream_t st) {
  rmsnorm_w_kernel<<<T, kNormThreads, 0, st>>>(h, w, H, eps, x);
  return cudaGetLastError();
}

}  // namespace fmoe
