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
constexpr uint32_t kErrWaitTimeout = 1u;   // a wait on words of other blocks (or a counter) ran out
constexpr uint32_t kErrCopyTimeout = 2u;   // bulk-copy barrier wait ran out
constexpr uint32_t kErrBadExpert = 4u;     // expert id outside [0, E)
constexpr uint32_t kErrRange = 8u;         // a partial sum outside the fixed-point range (|v| > 2^19)

// ---------------------------------------------------------------------------
// blob layout (the library's own statement of the packed format)
// ---------------------------------------------------------------------------
struct BlobLayout {
  size_t qh, sh;     // bytes of one gate/up row's codes and of its (scale,bias) words
  size_t gu_row;     // stride of gate/up row records [gate_q | up_q | gate_sb | up_sb], 16-byte padded
  size_t dq_off;     // offset of down column 0 (256-byte aligned)
  size_t dcol;       // bytes of one down column: H codes packed over rows (H*bits/8)
  size_t dsb_off;    // offset of the down (scale,bias) words of group 0 (256-byte aligned)
  size_t dsb_group;  // bytes of one group's down (scale,bias) words: one word per row (H*4)
  size_t bytes;      // blob size, a multiple of 256
};

__host__ __device__ inline size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

__host__ __device__ inline BlobLayout blob_layout(int bits, int H, int I) {
  BlobLayout L;
  L.qh = (size_t)H * bits / 8;
  L.sh = (size_t)H / kGroup * 4;
  L.gu_row = round_up(2 * L.qh + 2 * L.sh, 16);
  L.dq_off = round_up((size_t)I * L.gu_row, kPlaneAlign);
  L.dcol = (size_t)H * bits / 8;
  L.dsb_off = round_up(L.dq_off + (size_t)I * L.dcol, kPlaneAlign);
  L.dsb_group = (size_t)H * 4;
  L.bytes = round_up(L.dsb_off + (size_t)(I / kGroup) * L.dsb_group, kPlaneAlign);
  return L;
}

// ---------------------------------------------------------------------------
// workspace layout
// ---------------------------------------------------------------------------
struct WsLayout {
  size_t err;        // uint32 error word; the 256-byte header also holds:
  size_t exit_ctr;   //   uint32: blocks of the current launch that have finished
  size_t lbase;      //   uint32: layers run on this workspace, modulo 3 (picks the accumulator)
  size_t header_clear;  // bytes of the header a fresh call may zero (error word and exit count)
  size_t acc;        // u64 [3][H]: fixed-point (sum, count) accumulators of the persistent kernel
  size_t state;      // bytes at the start that are state kept between calls (header + acc)
  size_t ids;        // int32 [T][K]
  size_t weights;    // fp32 [T][K]
  size_t gate;       // fp32 [T]
  size_t h;          // fp32 [T][K+S][I]
  size_t y;          // fp32 [T][K+S][H] unweighted expert outputs (batched path)
  size_t xn;         // fp32 [H] normalised layer input (general path of a stack)
  size_t plan;       // int32 batch plan: 8-word header + 8 words per item
  size_t plan_words;
  size_t bytes;
};

inline WsLayout ws_layout(int H, int I, int S, int T, int K, int L) {
  (void)L;
  WsLayout w;
  size_t pos = 0;
  w.err = 0;
  w.exit_ctr = 96;
  w.lbase = 128;
  w.header_clear = 128;
  pos = 256;
  w.acc = pos; pos = round_up(pos + (size_t)3 * H * 8, 256);
  w.state = pos;
  w.ids = pos; pos = round_up(pos + (size_t)T * K * 4, 256);
  w.weights = pos; pos = round_up(pos + (size_t)T * K * 4, 256);
  w.gate = pos; pos = round_up(pos + (size_t)T * 4, 256);
  w.h = pos; pos = round_up(pos + (size_t)T * (K + S) * I * 4, 256);
  w.y = pos; pos = round_up(pos + (size_t)T * (K + S) * H * 4, 256);
  w.xn = pos; pos = round_up(pos + (size_t)H * 4, 256);
  // plan: header, then at most T*K + S*T items of 8 words (one token per
  // item at worst)
  w.plan_words = 8 + 8 * ((size_t)T * K + (size_t)S * T);
  w.plan = pos; pos = round_up(pos + w.plan_words * 4, 256);
  w.bytes = pos;
  return w;
}

// ---------------------------------------------------------------------------
// fixed-point partial sums
//
// Partial output sums of different blocks are added with 64-bit integer
// atomics, so the total does not depend on the order in which they arrive:
// a word holds (sum of round(v * 2^28)) << 8 plus, in its low 8 bits, the
// number of contributions (at most 255 contributors, so the count never
// carries into the sum).  |v| <= 2^19 per contribution keeps the sum of 255
// contributions inside the 56-bit signed field.
// ---------------------------------------------------------------------------
constexpr int kFixFrac = 28;
constexpr float kFixMax = 524288.0f;   // 2^19
constexpr int kFixCountBits = 8;
constexpr int kFixMaxContrib = (1 << kFixCountBits) - 1;

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

// 1 / pos_scale(i), exactly (a power of two).
template <int BITS>
__device__ __forceinline__ float inv_pos_scale(int i) {
  const int p = (BITS == 4) ? (i & 3) : (i & 7);
  const int e = 149 - kXScaleExp - BITS * p;                // 85 - BITS*p
  return __uint_as_float((uint32_t)(127 - e) << 23);
}

// The 32 inputs of a slice, pre-scaled by pos_scale, as 16 pairs (element
// 2k in .x, 2k+1 in .y) so that each packed fp32x2 FMA takes one pair.
typedef float2 SliceX[kSlice / 2];

template <int BITS> struct SliceCodes;
template <> struct SliceCodes<4> { uint4 v; };
template <> struct SliceCodes<2> { uint2 v; };

// A code masked in place, read as an fp32 (see the file comment).
__device__ __forceinline__ float mk(uint32_t w, uint32_t m) { return __uint_as_float(w & m); }
__device__ __forceinline__ float2 mk2(uint32_t w, uint32_t m0, uint32_t m1) { return make_float2(mk(w, m0), mk(w, m1)); }

// Sum over one 32-code slice of code * xs: returns 2^-64 * sum q_i x_i.
// Two independent packed accumulators; one AND per code, one fma.rn.f32x2
// per two codes.
__device__ __forceinline__ float slice_dot(const SliceCodes<4>& q, const SliceX& xs) {
  float2 a = make_float2(0.f, 0.f), c = make_float2(0.f, 0.f);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t w = (&q.v.x)[j];
    const uint32_t hi = w >> 16;
    a = __ffma2_rn(mk2(w, 0xFu, 0xF0u), xs[4 * j + 0], a);
    c = __ffma2_rn(mk2(w, 0xF00u, 0xF000u), xs[4 * j + 1], c);
    a = __ffma2_rn(mk2(hi, 0xFu, 0xF0u), xs[4 * j + 2], a);
    c = __ffma2_rn(mk2(hi, 0xF00u, 0xF000u), xs[4 * j + 3], c);
  }
  const float2 s = __fadd2_rn(a, c);
  return s.x + s.y;
}

__device__ __forceinline__ float slice_dot(const SliceCodes<2>& q, const SliceX& xs) {
  float2 a = make_float2(0.f, 0.f), c = make_float2(0.f, 0.f);
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const uint32_t w = (&q.v.x)[j];
    const uint32_t hi = w >> 16;
    a = __ffma2_rn(mk2(w, 0x3u, 0xCu), xs[8 * j + 0], a);
    c = __ffma2_rn(mk2(w, 0x30u, 0xC0u), xs[8 * j + 1], c);
    a = __ffma2_rn(mk2(w, 0x300u, 0xC00u), xs[8 * j + 2], a);
    c = __ffma2_rn(mk2(w, 0x3000u, 0xC000u), xs[8 * j + 3], c);
    a = __ffma2_rn(mk2(hi, 0x3u, 0xCu), xs[8 * j + 4], a);
    c = __ffma2_rn(mk2(hi, 0x30u, 0xC0u), xs[8 * j + 5], c);
    a = __ffma2_rn(mk2(hi, 0x300u, 0xC00u), xs[8 * j + 6], a);
    c = __ffma2_rn(mk2(hi, 0x3000u, 0xC000u), xs[8 * j + 7], c);
  }
  const float2 s = __fadd2_rn(a, c);
  return s.x + s.y;
}

// Contribution of one slice to a row dot product:
//   s * sum q x + b * sum x  over the slice's 32 columns,
// where sb is the (scale, bias) word of the slice's group and xsum is the
// plain sum of the slice's 32 (unscaled) inputs.
template <int BITS>
__device__ __forceinline__ float slice_term(const SliceCodes<BITS>& q, uint32_t sb, const SliceX& xs,
                                            float xsum) {
  const float p = slice_dot(q, xs);
  const float s64 = bf16lo(sb) * 18446744073709551616.0f;   // scale * 2^64
  return fmaf(s64, p, bf16hi(sb) * xsum);
}

// Pre-scale four consecutive inputs (elements 4j..4j+3 of a slice) into the
// pair array; returns their plain sum.
template <int BITS>
__device__ __forceinline__ float put_x4(SliceX& xs, int j, float4 v) {
  xs[2 * j] = make_float2(v.x * pos_scale<BITS>(4 * j + 0), v.y * pos_scale<BITS>(4 * j + 1));
  xs[2 * j + 1] = make_float2(v.z * pos_scale<BITS>(4 * j + 2), v.w * pos_scale<BITS>(4 * j + 3));
  return (v.x + v.y) + (v.z + v.w);
}

// Load the 32 inputs of slice `s` from fp32 global memory, multiplied by
// `scale` and pre-scaled; returns the plain sum of the scaled values.  `CG`
// selects an L2-only load (data written earlier in the same kernel by other
// blocks).
template <int BITS, bool CG>
__device__ __forceinline__ float load_slice_x(const float* __restrict__ x, int s, float scale, SliceX& xs) {
  const float4* p = reinterpret_cast<const float4*>(x + (size_t)s * kSlice);
  float sum = 0.f;
#pragma unroll
  for (int j = 0; j < kSlice / 4; ++j) {
    float4 v = CG ? __ldcg(p + j) : __ldg(p + j);
    v.x *= scale; v.y *= scale; v.z *= scale; v.w *= scale;
    sum += put_x4<BITS>(xs, j, v);
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

// Top-K key of a logit: an unsigned integer whose order is the order of the
// fp32 values (larger = larger logit), -0 and +0 mapped to the same key.
// Valid keys are never 0.
__device__ __forceinline__ uint32_t logit_key(float v) {
  uint32_t b = __float_as_uint(v);
  if (b == 0x80000000u) b = 0u;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// The fp32 value of a logit_key.
__device__ __forceinline__ float key_logit(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// Top-K of E logits, executed by one full warp.  Each lane keeps its best
// remaining key; a round takes the warp maximum (redux.sync), the lowest id
// holding it, and that lane rescans.  Lane k < K receives the k-th pick
// (descending logit, equal logits -> lower id) and its logit in (my_id,
// my_l); other lanes get (-1, 0).  E <= 1024.
__device__ __forceinline__ void warp_topk(const float* __restrict__ logits, int E, int K, int& my_id,
                                          float& my_l) {
  const int lane = threadIdx.x & 31;
  const int nv = (E + 31) >> 5;
  uint32_t key[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const int id = lane + 32 * j;
    key[j] = (j < nv && id < E) ? logit_key(__ldg(logits + id)) : 0u;
  }
  uint32_t bk = 0u;
  int bj = 0;
#pragma unroll
  for (int j = 0; j < 32; ++j)
    if (key[j] > bk) {
      bk = key[j];
      bj = j;
    }
  my_l = 0.f;
  my_id = -1;
  for (int k = 0; k < K; ++k) {
    const uint32_t m = __reduce_max_sync(0xFFFFFFFFu, bk);
    const uint32_t cid = __reduce_min_sync(0xFFFFFFFFu, bk == m ? (uint32_t)(lane + 32 * bj) : 0xFFFFFFFFu);
    if (lane == k) {
      my_l = key_logit(m);
      my_id = (int)cid;
    }
    if ((int)(cid & 31u) == lane) {        // the winner's lane drops it and rescans
      const int jr = (int)(cid >> 5);
      bk = 0u;
      bj = 0;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        if (j == jr) key[j] = 0u;
        if (key[j] > bk) {
          bk = key[j];
          bj = j;
        }
      }
    }
  }
}

// Softmax over the K picks of warp_topk (lane k < K holds pick k's logit):
// the weight of lane k's pick, 0 on other lanes.
__device__ __forceinline__ float warp_topk_softmax(float my_l, int K) {
  const int lane = threadIdx.x & 31;
  const float lmax = __shfl_sync(0xFFFFFFFFu, my_l, 0);
  const float e = (lane < K) ? expf(my_l - lmax) : 0.f;
  const float tot = warp_sum(e);
  return (lane < K) ? e / tot : 0.f;
}

// Top-K + softmax over the selected logits (flash-moe write-up, "per-layer
// pipeline": softmax + top-K routing); one full warp.
__device__ __forceinline__ void warp_route(const float* __restrict__ logits, int E, int K,
                                           int& my_id, float& my_w) {
  float my_l;
  warp_topk(logits, E, K, my_id, my_l);
  my_w = warp_topk_softmax(my_l, K);
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

// One contribution to a fixed-point accumulator word (see above); a value
// outside the range is clamped and reported.
__device__ __forceinline__ unsigned long long fix_word(float v, uint32_t* err) {
  if (!(fabsf(v) <= kFixMax)) {     // also catches NaN
    atomicOr(err, kErrRange);
    v = (v != v) ? 0.f : copysignf(kFixMax, v);
  }
  const long long q = __float2ll_rn(v * (float)(1 << kFixFrac));
  return ((unsigned long long)q << kFixCountBits) + 1ull;
}

__device__ __forceinline__ int fix_count(unsigned long long w) { return (int)(w & ((1u << kFixCountBits) - 1)); }

__device__ __forceinline__ float fix_value(unsigned long long w) {
  return __ll2float_rn((long long)w >> kFixCountBits) * (1.0f / (float)(1 << kFixFrac));
}

__device__ __forceinline__ void red_add_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("red.relaxed.gpu.global.add.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ void signal_counter(uint32_t* ctr) {
  __threadfence();
  atomicAdd(ctr, 1u);
}

}  // namespace fmoe
