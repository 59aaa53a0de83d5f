// Internal device helpers of libfmoe (sm_103a).
//
// The expert weights are affine group-quantised codes (flash-moe write-up,
// discuss.pytorch.kr, section "FMA-optimised dequant kernel": weight =
// nibble * scale + bias).  The kernels never materialise dequantised weights:
// for every 64-column group g of a row they use
//     sum_c (q_c s_g + b_g) x_c = s_g * sum_c q_c x_c + b_g * sum_c x_c,
// the write-up's "precompute scale*x and bias*x" idea taken per group, so the
// inner loop is one fused multiply-add per code.
//
// Code extraction without an int->float conversion: masking a code in place
// (w & (0xF << 4p)) leaves an integer below 2^24 whose bit pattern, read as
// an fp32, is exactly q * 2^(4p) * 2^-149 (a subnormal, or the smallest
// normal binade, where the value is the integer times 2^-149).  The matching
// input is pre-scaled once per token by 2^(149 - 4p - 64), so each product
// is q * x * 2^-64 exactly as an fp32 product would be, and the group sum is
// rescaled by 2^64 when it meets the scale.  Subnormal operands are handled
// at full rate by the FMA pipes as long as flush-to-zero is off (the library
// is built with -ftz=false and the inline PTX below never uses .ftz).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/fmoe.h"

namespace fmoe {

constexpr int kGroup = 64;
constexpr int kPlaneAlign = 256;
constexpr int kSlice = 32;            // codes per lane slice (16 B at 4-bit, 8 B at 2-bit)
constexpr int kXScaleExp = 64;        // products carry a factor 2^-64

// error-word bits
constexpr uint32_t kErrWaitTimeout = 1u;   // device-wide counter wait ran out
constexpr uint32_t kErrCopyTimeout = 2u;   // bulk-copy barrier wait ran out
constexpr uint32_t kErrBadExpert = 4u;     // expert id outside [0, E)

// ---------------------------------------------------------------------------
// blob layout (the library's own statement of the packed format)
// ---------------------------------------------------------------------------
struct BlobLayout {
  size_t gate_q, gate_sb, up_q, up_sb, down_q, down_sb, bytes;
};

__host__ __device__ inline size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

__host__ __device__ inline BlobLayout blob_layout(int bits, int H, int I) {
  BlobLayout L;
  const size_t qrow_in_h = (size_t)H * bits / 8;   // bytes of one gate/up code row
  const size_t sbrow_in_h = (size_t)H / kGroup * 4;
  const size_t qrow_in_i = (size_t)I * bits / 8;   // bytes of one down code row
  const size_t sbrow_in_i = (size_t)I / kGroup * 4;
  size_t pos = 0;
  L.gate_q = pos;  pos = round_up(pos + (size_t)I * qrow_in_h, kPlaneAlign);
  L.gate_sb = pos; pos = round_up(pos + (size_t)I * sbrow_in_h, kPlaneAlign);
  L.up_q = pos;    pos = round_up(pos + (size_t)I * qrow_in_h, kPlaneAlign);
  L.up_sb = pos;   pos = round_up(pos + (size_t)I * sbrow_in_h, kPlaneAlign);
  L.down_q = pos;  pos = round_up(pos + (size_t)H * qrow_in_i, kPlaneAlign);
  L.down_sb = pos; pos = round_up(pos + (size_t)H * sbrow_in_i, kPlaneAlign);
  L.bytes = pos;
  return L;
}

// ---------------------------------------------------------------------------
// workspace layout
// ---------------------------------------------------------------------------
struct WsLayout {
  size_t err;        // uint32 error word (+ padding)
  size_t counters;   // uint32 device-wide counters
  size_t n_counters;
  size_t ids;        // int32 [T][K]
  size_t weights;    // fp32 [T][K]
  size_t gate;       // fp32 [T]
  size_t h;          // fp32 [T][K+S][I]
  size_t hbuf;       // fp32 [2][H] stack ping-pong
  size_t plan;       // int32 batch plan
  size_t plan_words;
  size_t bytes;
};

inline WsLayout ws_layout(int H, int I, int S, int T, int K, int L) {
  WsLayout w;
  size_t pos = 0;
  w.err = pos; pos += 256;
  w.counters = pos;
  // per layer: one counter per slot, one layer-done counter; plus exit/test counters
  w.n_counters = (size_t)L * (K + S + 1) + 8;
  pos = round_up(pos + w.n_counters * 4, 256);
  w.ids = pos; pos = round_up(pos + (size_t)T * K * 4, 256);
  w.weights = pos; pos = round_up(pos + (size_t)T * K * 4, 256);
  w.gate = pos; pos = round_up(pos + (size_t)T * 4, 256);
  w.h = pos; pos = round_up(pos + (size_t)T * (K + S) * I * 4, 256);
  w.hbuf = pos; pos = round_up(pos + (size_t)2 * H * 4, 256);
  // plan: unique count, unique ids[T*K+1], per-unique token count, token lists
  w.plan_words = 4 + 4 * (size_t)(T * K + 1) + (size_t)(T * K + 1) * (T + 1);
  w.plan = pos; pos = round_up(pos + w.plan_words * 4, 256);
  w.bytes = pos;
  return w;
}

// ---------------------------------------------------------------------------
// small device helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float bf16v(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// d.xy += a.xy * b.xy with one packed fp32x2 FMA (round to nearest, subnormals kept)
__device__ __forceinline__ void ffma2(float& d0, float& d1, float a0, float a1, float b0, float b1) {
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\t"
      "mov.b64 rb, {%4, %5};\n\t"
      "mov.b64 rd, {%0, %1};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rd;\n\t"
      "mov.b64 {%0, %1}, rd;\n\t}"
      : "+f"(d0), "+f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

// Positional pre-scale of input element i of a 32-code slice.
//   4-bit: codes 0..3 of a word are masked from the word, codes 4..7 from
//          the word shifted right by 16; position p = i mod 4, factor 2^(85-4p)
//   2-bit: codes 0..7 from the word, 8..15 from word >> 16; p = i mod 8,
//          factor 2^(85-2p)
template <int BITS>
__device__ __forceinline__ float pos_scale(int i) {
  const int p = (BITS == 4) ? (i & 3) : (i & 7);
  const int e = 149 - kXScaleExp - BITS * p;                // 85 - BITS*p
  return __uint_as_float((uint32_t)(e + 127) << 23);
}

// Sum over one 32-code slice of code * xs (xs pre-scaled by pos_scale):
// returns 2^-64 * sum q_i x_i.
template <int BITS> struct SliceCodes;
template <> struct SliceCodes<4> { uint4 v; };
template <> struct SliceCodes<2> { uint2 v; };

__device__ __forceinline__ float mk(uint32_t w, uint32_t m) { return __uint_as_float(w & m); }

__device__ __forceinline__ float slice_dot(const SliceCodes<4>& q, const float (&xs)[kSlice]) {
  float a0 = 0.f, a1 = 0.f, c0 = 0.f, c1 = 0.f;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t w = (&q.v.x)[j];
    const uint32_t hi = w >> 16;
    const float* x = xs + 8 * j;
    if (j & 1) {
      ffma2(c0, c1, mk(w, 0xFu), mk(w, 0xF0u), x[0], x[1]);
      ffma2(c0, c1, mk(w, 0xF00u), mk(w, 0xF000u), x[2], x[3]);
      ffma2(c0, c1, mk(hi, 0xFu), mk(hi, 0xF0u), x[4], x[5]);
      ffma2(c0, c1, mk(hi, 0xF00u), mk(hi, 0xF000u), x[6], x[7]);
    } else {
      ffma2(a0, a1, mk(w, 0xFu), mk(w, 0xF0u), x[0], x[1]);
      ffma2(a0, a1, mk(w, 0xF00u), mk(w, 0xF000u), x[2], x[3]);
      ffma2(a0, a1, mk(hi, 0xFu), mk(hi, 0xF0u), x[4], x[5]);
      ffma2(a0, a1, mk(hi, 0xF00u), mk(hi, 0xF000u), x[6], x[7]);
    }
  }
  return (a0 + a1) + (c0 + c1);
}

__device__ __forceinline__ float slice_dot(const SliceCodes<2>& q, const float (&xs)[kSlice]) {
  float a0 = 0.f, a1 = 0.f, c0 = 0.f, c1 = 0.f;
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const uint32_t w = (&q.v.x)[j];
    const uint32_t hi = w >> 16;
    const float* x = xs + 16 * j;
    ffma2(a0, a1, mk(w, 0x3u), mk(w, 0xCu), x[0], x[1]);
    ffma2(c0, c1, mk(w, 0x30u), mk(w, 0xC0u), x[2], x[3]);
    ffma2(a0, a1, mk(w, 0x300u), mk(w, 0xC00u), x[4], x[5]);
    ffma2(c0, c1, mk(w, 0x3000u), mk(w, 0xC000u), x[6], x[7]);
    ffma2(a0, a1, mk(hi, 0x3u), mk(hi, 0xCu), x[8], x[9]);
    ffma2(c0, c1, mk(hi, 0x30u), mk(hi, 0xC0u), x[10], x[11]);
    ffma2(a0, a1, mk(hi, 0x300u), mk(hi, 0xC00u), x[12], x[13]);
    ffma2(c0, c1, mk(hi, 0x3000u), mk(hi, 0xC000u), x[14], x[15]);
  }
  return (a0 + a1) + (c0 + c1);
}

// Contribution of one slice to a row dot product:
//   s * sum q x + b * sum x  over the slice's 32 columns,
// where sb is the (scale, bias) word of the slice's group and xsum is the
// plain sum of the slice's 32 (unscaled) inputs.
template <int BITS>
__device__ __forceinline__ float slice_term(const SliceCodes<BITS>& q, uint32_t sb,
                                            const float (&xs)[kSlice], float xsum) {
  const float p = slice_dot(q, xs);
  const float s64 = bf16lo(sb) * 18446744073709551616.0f;   // scale * 2^64
  return fmaf(s64, p, bf16hi(sb) * xsum);
}

// Load the 32 inputs of slice `s` from fp32 global memory, pre-scaled; returns
// their plain sum.  `cg` selects an L2-only load (data written earlier in the
// same kernel by other blocks).
template <int BITS, bool CG>
__device__ __forceinline__ float load_slice_x(const float* __restrict__ x, int s, float scale,
                                              float (&xs)[kSlice]) {
  const float4* p = reinterpret_cast<const float4*>(x + (size_t)s * kSlice);
  float sum = 0.f;
#pragma unroll
  for (int j = 0; j < kSlice / 4; ++j) {
    float4 v = CG ? __ldcg(p + j) : __ldg(p + j);
    v.x *= scale; v.y *= scale; v.z *= scale; v.w *= scale;
    sum += (v.x + v.y) + (v.z + v.w);
    xs[4 * j + 0] = v.x * pos_scale<BITS>(4 * j + 0);
    xs[4 * j + 1] = v.y * pos_scale<BITS>(4 * j + 1);
    xs[4 * j + 2] = v.z * pos_scale<BITS>(4 * j + 2);
    xs[4 * j + 3] = v.w * pos_scale<BITS>(4 * j + 3);
  }
  return sum;
}

__device__ __forceinline__ float warp_sum(float v, int width = 32) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1)
    if (o < width) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

__device__ __forceinline__ float silu_f(float a) { return a / (1.0f + expf(-a)); }
__device__ __forceinline__ float sigmoid_f(float z) { return 1.0f / (1.0f + expf(-z)); }

// "a ranks before b": larger logit first, equal logits -> lower id first.
// Float comparison treats -0 and +0 as equal.
__device__ __forceinline__ bool ranks_before(float av, int ai, float bv, int bi) {
  return av > bv || (av == bv && ai < bi);
}

// Top-K of E logits + softmax over the selected ones; executed by one full
// warp (flash-moe write-up, "per-layer pipeline": softmax + top-K routing).
// Lane k < K receives the k-th pick in (*id_out, *w_out) of its own lane;
// the function returns (id, weight) for lanes < K and (-1, 0) otherwise.
// E <= 1024.
__device__ __forceinline__ void warp_route(const float* __restrict__ logits, int E, int K,
                                           int& my_id, float& my_w) {
  const int lane = threadIdx.x & 31;
  float v[32];
  uint32_t taken = 0;
  const int nv = (E + 31) >> 5;
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] = (j < nv && lane + 32 * j < E) ? __ldg(logits + lane + 32 * j) : 0.f;
  // local best
  auto local_best = [&](float& bv, int& bi) {
    bv = 0.f; bi = 0x7FFFFFFF;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const int id = lane + 32 * j;
      if (j < nv && id < E && !((taken >> j) & 1u)) {
        if (bi == 0x7FFFFFFF || ranks_before(v[j], id, bv, bi)) { bv = v[j]; bi = id; }
      }
    }
  };
  float bv; int bi;
  local_best(bv, bi);
  my_id = -1;
  float my_l = 0.f;
  for (int k = 0; k < K; ++k) {
    float cv = bv; int ci = bi;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
      const float ov = __shfl_xor_sync(0xFFFFFFFFu, cv, o);
      const int oi = __shfl_xor_sync(0xFFFFFFFFu, ci, o);
      if (oi != 0x7FFFFFFF && (ci == 0x7FFFFFFF || ranks_before(ov, oi, cv, ci))) { cv = ov; ci = oi; }
    }
    if (lane == k) { my_id = ci; my_l = cv; }
    if ((ci & 31) == lane) {            // the winner's lane drops it and rescans
      taken |= 1u << (ci >> 5);
      local_best(bv, bi);
    }
  }
  const float lmax = __shfl_sync(0xFFFFFFFFu, my_l, 0);
  const float e = (lane < K) ? expf(my_l - lmax) : 0.f;
  const float tot = warp_sum(e);
  my_w = (lane < K) ? e / tot : 0.f;
}

// Wait until *ctr >= target, for at most timeout_ns; on time-out set the error
// bit and return false.  Called by one thread.
__device__ __forceinline__ bool wait_counter(const uint32_t* ctr, uint32_t target, uint64_t timeout_ns,
                                             uint32_t* err) {
  const uint64_t t0 = global_timer_ns();
  while (true) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
    if (v >= target) return true;
    if (global_timer_ns() - t0 > timeout_ns) {
      atomicOr(err, kErrWaitTimeout);
      return false;
    }
    __nanosleep(64);
  }
}

__device__ __forceinline__ void signal_counter(uint32_t* ctr) {
  __threadfence();
  atomicAdd(ctr, 1u);
}

}  // namespace fmoe
