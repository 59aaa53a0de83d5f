// Routing kernel and the batched (T >= 1 tokens) expert kernels.
//
// The single-launch persistent kernel (fmoe_fused.cu) is the fast path for one
// token; these kernels serve every shape the ABI accepts at any T, and read
// each DISTINCT expert of a batch once: when several tokens pick the same
// expert, its codes are dequantised once per 32-column slice and applied to
// all of those tokens from registers.  The write-ups stream experts for one
// token at a time; their failed-experiments table notes that per-token expert
// I/O is what makes batching (speculative decoding) pay nothing, which is the
// cost this deduplication removes for resident experts.
//
// Sequence (four launches on one stream, graph-capturable):
//   batch_plan_kernel    route (top-K + softmax, shared gate) or take given
//                        ids; list the distinct experts and, for each, the
//                        tokens that picked it, in groups of G <= 4
//   batch_gateup_kernel  h[t][k] = silu(Wg x_t) * (Wu x_t) for every (expert,
//                        token group) item, 2 intermediate rows per warp
//   batch_down_kernel    y[t][k] = Wd h[t][k]; a unit is 256 (4-bit) or 512
//                        (2-bit) output rows, the down projection being
//                        stored by column (tensor-map tiles of column slices)
//   batch_combine_kernel out[t] = residual[t] + sum_k w[t][k] y[t][k] + g[t] y[t][K]
// The two expert kernels run one block per SM over a contiguous share of
// (item, row block) work units.  In the gate/up kernel a producer warp
// streams each unit's packed rows (one contiguous range of the blob) into a
// shared-memory ring with bulk asynchronous copies (TMA engine, mbarrier
// completion) and eight consumer warps compute from the ring; the down
// kernel's producer streams tiles of column slices with tensor copies.
//
// Sources: flash-moe write-up (discuss.pytorch.kr): "per-layer pipeline"
// (softmax + top-K routing, expert forward, combine), "hand-written Metal
// compute shaders" (dequant matvec, fused SwiGLU, MoE combine + residual +
// sigmoid gate), "FMA-optimised dequant kernel" (code * scale + bias).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "fmoe_async.cuh"
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
      // eight columns per lane and step (H is a multiple of 64)
      const uint4* w8 = reinterpret_cast<const uint4*>(wsg);
      const float4* x4 = reinterpret_cast<const float4*>(x + (size_t)t * H);
      for (int c = lane; c < H / 8; c += 32) {
        const uint4 wb = __ldg(w8 + c);
        const float4 a = __ldg(x4 + 2 * c), b = __ldg(x4 + 2 * c + 1);
        acc += (bf16lo(wb.x) * a.x + bf16hi(wb.x) * a.y) + (bf16lo(wb.y) * a.z + bf16hi(wb.y) * a.w);
        acc += (bf16lo(wb.z) * b.x + bf16hi(wb.z) * b.y) + (bf16lo(wb.w) * b.z + bf16hi(wb.w) * b.w);
      }
      acc = warp_sum(acc);
    }
    if (lane == 0) gate[t] = (wsg != nullptr) ? sigmoid_f(acc) : 0.f;
  }
}

// ---------------------------------------------------------------------------
// plan: distinct experts and their token groups
// ---------------------------------------------------------------------------
constexpr int kPlanThreads = 512;
constexpr int kPlanWarps = kPlanThreads / 32;
constexpr int kMaxPairs = FMOE_MAX_TOKENS * FMOE_MAX_TOPK;
static_assert(kMaxPairs <= kPlanThreads, "one thread per (token, slot) pair");
static_assert(FMOE_MAX_TOKENS <= kPlanWarps, "one warp per token");
static_assert(kPlanHeader == 8 && kItemWords == 8, "ws_layout sizes the plan for these");

// Relative cost of one work unit of an item with n tokens: its bytes (a
// constant per unit) plus its arithmetic (one pass per token).
__device__ __forceinline__ int unit_cost(int n) { return 2 + n; }

// Item i of the plan (kItemWords int32 at plan + kPlanHeader + i * kItemWords):
//   [0] expert id (-1: the shared expert)   [1] n tokens (1..G)
//   [2 + g] (t << 8) | slot of the g-th token: h[t][slot] / y[t][slot]
//   [6] sum of unit_cost over the items before i
// Header: [0] items, [1] distinct experts (shared included), [2] cost total.
__global__ void __launch_bounds__(kPlanThreads) batch_plan_kernel(BatchArgs a) {
  __shared__ int s_id[kMaxPairs];
  __shared__ int s_rank[kMaxPairs];   // earlier pairs with the same expert
  __shared__ int s_cnt[kMaxPairs];    // all pairs with the same expert
  __shared__ int s_first[kMaxPairs];  // first pair with the same expert
  __shared__ int s_base[kMaxPairs];   // first item of the expert (valid at first pairs)
  __shared__ float s_gpart[kPlanWarps][FMOE_MAX_TOKENS];
  __shared__ int s_nitems, s_nuniq;
  __shared__ int s_itemn[kMaxPairs + FMOE_MAX_TOKENS];   // tokens of each item
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int T = a.T, K = a.K, NS = a.K + a.S, TK = a.T * a.K, G = a.geo.G;

  if (a.logits != nullptr) {
    if (warp < T) {
      int id; float w;
      warp_route(a.logits + (size_t)warp * a.E, a.E, K, id, w);
      if (lane < K) {
        a.ids[warp * K + lane] = id;
        a.weights[warp * K + lane] = w;
        s_id[warp * K + lane] = id;
      }
    }
    if (a.S) {
      // w_sg . x_t for every token: warp w takes a sixteenth of the columns
      // of all tokens, eight tokens at a time with all their loads in flight
      constexpr int kTokChunk = 8;
      const int H4 = a.H / 4, per = (H4 + kPlanWarps - 1) / kPlanWarps;
      const int c0 = warp * per, c1 = min(H4, c0 + per);
      const uint2* w4 = reinterpret_cast<const uint2*>(a.wsg);
      const float4* x4 = reinterpret_cast<const float4*>(a.x);
      for (int t0 = 0; t0 < T; t0 += kTokChunk) {
        float acc[kTokChunk];
#pragma unroll
        for (int t = 0; t < kTokChunk; ++t) acc[t] = 0.f;
        for (int c = c0 + lane; c < c1; c += 64) {
          const bool two = c + 32 < c1;
          const uint2 wa = __ldg(w4 + c);
          const uint2 wb = two ? __ldg(w4 + c + 32) : make_uint2(0u, 0u);
          float4 xa[kTokChunk], xb[kTokChunk];
#pragma unroll
          for (int t = 0; t < kTokChunk; ++t) {
            const bool in = t0 + t < T;
            xa[t] = in ? __ldcg(x4 + (size_t)(t0 + t) * H4 + c) : make_float4(0.f, 0.f, 0.f, 0.f);
            xb[t] = (in && two) ? __ldcg(x4 + (size_t)(t0 + t) * H4 + c + 32) : make_float4(0.f, 0.f, 0.f, 0.f);
          }
#pragma unroll
          for (int t = 0; t < kTokChunk; ++t) {
            acc[t] = fmaf(bf16lo(wa.x), xa[t].x, acc[t]);
            acc[t] = fmaf(bf16hi(wa.x), xa[t].y, acc[t]);
            acc[t] = fmaf(bf16lo(wa.y), xa[t].z, acc[t]);
            acc[t] = fmaf(bf16hi(wa.y), xa[t].w, acc[t]);
            acc[t] = fmaf(bf16lo(wb.x), xb[t].x, acc[t]);
            acc[t] = fmaf(bf16hi(wb.x), xb[t].y, acc[t]);
            acc[t] = fmaf(bf16lo(wb.y), xb[t].z, acc[t]);
            acc[t] = fmaf(bf16hi(wb.y), xb[t].w, acc[t]);
          }
        }
#pragma unroll
        for (int t = 0; t < kTokChunk; ++t) {
          const float v = warp_sum(acc[t]);
          if (lane == 0 && t0 + t < T) s_gpart[warp][t0 + t] = v;
        }
      }
    }
  } else {
    for (int p = tid; p < TK; p += kPlanThreads) {
      int id = a.ids_in[p];
      if (id < 0 || id >= a.E) {
        atomicOr(a.err, kErrBadExpert);
        id = -1;
      }
      s_id[p] = id;
    }
  }
  __syncthreads();

  if (a.logits != nullptr && a.S && tid < T) {
    float g = 0.f;
    for (int w = 0; w < kPlanWarps; ++w) g += s_gpart[w][tid];
    a.gate[tid] = sigmoid_f(g);
  }

  // an expert id outside [0, E) leaves its output row zero
  if (a.ids_in != nullptr) {
    for (int p = 0; p < TK; ++p)
      if (s_id[p] < 0) {
        float* yrow = a.y + ((size_t)(p / K) * NS + (p % K)) * a.H;
        for (int j = tid; j < a.H; j += kPlanThreads) yrow[j] = 0.f;
      }
  }

  if (tid < TK) {
    const int id = s_id[tid];
    int rank = 0, cnt = 0, first = tid;
    if (id >= 0) {
      for (int q = 0; q < TK; ++q) {
        if (s_id[q] == id) {
          ++cnt;
          if (q < tid) ++rank;
          if (q < first) first = q;
        }
      }
    }
    s_rank[tid] = rank;
    s_cnt[tid] = cnt;
    s_first[tid] = first;
  }
  __syncthreads();

  // items of each distinct expert, in order of first appearance
  if (warp == 0) {
    int base = 0, uniq = 0;
    for (int c0 = 0; c0 < TK; c0 += 32) {
      const int p = c0 + lane;
      const bool lead = p < TK && s_id[p] >= 0 && s_rank[p] == 0;
      const int n = lead ? (s_cnt[p] + G - 1) / G : 0;
      int incl = n;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += v;
      }
      if (p < TK) s_base[p] = base + incl - n;
      base += __shfl_sync(0xFFFFFFFFu, incl, 31);
      uniq += __popc(__ballot_sync(0xFFFFFFFFu, lead));
    }
    if (lane == 0) {
      s_nitems = base;
      s_nuniq = uniq;
    }
  }
  __syncthreads();

  int32_t* items = a.plan + kPlanHeader;
  if (tid < TK && s_id[tid] >= 0) {
    const int r = s_rank[tid];
    const int it = s_base[s_first[tid]] + r / G;
    const int g = r % G;
    items[it * kItemWords + 2 + g] = ((tid / K) << 8) | (tid % K);
    if (g == 0) {
      items[it * kItemWords + 0] = s_id[tid];
      items[it * kItemWords + 1] = min(G, s_cnt[tid] - r);
      s_itemn[it] = min(G, s_cnt[tid] - r);
    }
  }
  const int n_shared_items = a.S ? (T + G - 1) / G : 0;
  if (a.S && tid < T) {
    const int it = s_nitems + tid / G;
    const int g = tid % G;
    items[it * kItemWords + 2 + g] = (tid << 8) | K;
    if (g == 0) {
      items[it * kItemWords + 0] = -1;
      items[it * kItemWords + 1] = min(G, T - tid);
      s_itemn[it] = min(G, T - tid);
    }
  }
  __syncthreads();
  // cost prefix of the items (item word 6) and the total (header word 2):
  // the expert kernels split their work units by cost, not by count
  const int n_items = s_nitems + n_shared_items;
  if (warp == 0) {
    int base = 0;
    for (int c0 = 0; c0 < n_items; c0 += 32) {
      const int i = c0 + lane;
      const int cst = i < n_items ? unit_cost(s_itemn[i]) : 0;
      int incl = cst;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += v;
      }
      if (i < n_items) items[i * kItemWords + 6] = base + incl - cst;
      base += __shfl_sync(0xFFFFFFFFu, incl, 31);
    }
    if (lane == 0) {
      a.plan[0] = n_items;
      a.plan[1] = s_nuniq + a.S;
      a.plan[2] = base;
    }
  }
}

// ---------------------------------------------------------------------------
// expert kernels: shared helpers
// ---------------------------------------------------------------------------
// Codes 8j..8j+7 of a 32-code slice (one "octet"), masked in place as the
// pairs (2i, 2i+1), i = 0..3, that meet the pre-scaled inputs.
__device__ __forceinline__ void octet_pairs(const SliceCodes<4>& q, int j, float2 (&p)[4]) {
  const uint32_t w = (&q.v.x)[j];
  const uint32_t hi = w >> 16;
  p[0] = mk2(w, 0xFu, 0xF0u);
  p[1] = mk2(w, 0xF00u, 0xF000u);
  p[2] = mk2(hi, 0xFu, 0xF0u);
  p[3] = mk2(hi, 0xF00u, 0xF000u);
}

__device__ __forceinline__ void octet_pairs(const SliceCodes<2>& q, int j, float2 (&p)[4]) {
  const uint32_t w = (&q.v.x)[j >> 1] >> (16 * (j & 1));
  p[0] = mk2(w, 0x3u, 0xCu);
  p[1] = mk2(w, 0x30u, 0xC0u);
  p[2] = mk2(w, 0x300u, 0xC00u);
  p[3] = mk2(w, 0x3000u, 0xC000u);
}

// The codes of slice s of a row held in shared memory.
template <int BITS>
__device__ __forceinline__ SliceCodes<BITS> smem_codes(const uint8_t* row, int s) {
  SliceCodes<BITS> q;
  if constexpr (BITS == 4) q.v = reinterpret_cast<const uint4*>(row)[s];
  else q.v = reinterpret_cast<const uint2*>(row)[s];
  return q;
}

// acc[r] += code[r] * h for the rows of one 32-bit code word of a down column
// (codes masked in place, h pre-scaled per position; hv: 2 pairs at 4-bit,
// 4 at 2-bit).
// The masked code pairs of one 32-bit word of a down column (RW/2 pairs of
// rows, each value carrying the position's power-of-two factor that the
// pre-scaled h of that position cancels).
template <int BITS>
__device__ __forceinline__ void code_pairs(uint32_t w, float2* q) {
  const uint32_t hi = w >> 16;
  if constexpr (BITS == 4) {
    q[0] = mk2(w, 0xFu, 0xF0u);
    q[1] = mk2(w, 0xF00u, 0xF000u);
    q[2] = mk2(hi, 0xFu, 0xF0u);
    q[3] = mk2(hi, 0xF00u, 0xF000u);
  } else {
    q[0] = mk2(w, 0x3u, 0xCu);
    q[1] = mk2(w, 0x30u, 0xC0u);
    q[2] = mk2(w, 0x300u, 0xC00u);
    q[3] = mk2(w, 0x3000u, 0xC000u);
    q[4] = mk2(hi, 0x3u, 0xCu);
    q[5] = mk2(hi, 0x30u, 0xC0u);
    q[6] = mk2(hi, 0x300u, 0xC00u);
    q[7] = mk2(hi, 0x3000u, 0xC000u);
  }
}

// Down step of `ncol` columns of a tile ([column][bx bytes], the lane's code
// word at word `lane` of each column) for NT tokens: acc[t] += codes * h, the
// codes masked once per column and met by every token from registers.  hq
// holds, per token and column, h times the position factors of positions
// 0..3 (positions 4..7 of a 2-bit word are those times 2^-8); hs[t] sums the
// position-0 values (h times a power of two).
template <int BITS, int NT>
__device__ __forceinline__ void bd_columns(const uint8_t* tile, int bx, int ncol, bool row_ok, const float4* hq, int I,
                                           float2 (&acc)[kMaxTokGroup][16 / BITS], float (&hs)[kMaxTokGroup]) {
  constexpr int P = 16 / BITS;
  const int lane = threadIdx.x & 31;
#pragma unroll 2
  for (int j = 0; j < ncol; ++j) {
    const uint32_t w = row_ok ? reinterpret_cast<const uint32_t*>(tile + (size_t)j * bx)[lane] : 0u;
    float2 q[P];
    code_pairs<BITS>(w, q);
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const float4 a = hq[(size_t)t * I + j];
      hs[t] += a.x;
      const float2 h01 = make_float2(a.x, a.y), h23 = make_float2(a.z, a.w);
      if constexpr (BITS == 4) {
        acc[t][0] = __ffma2_rn(q[0], h01, acc[t][0]);
        acc[t][1] = __ffma2_rn(q[1], h23, acc[t][1]);
        acc[t][2] = __ffma2_rn(q[2], h01, acc[t][2]);
        acc[t][3] = __ffma2_rn(q[3], h23, acc[t][3]);
      } else {
        const float2 k8 = make_float2(0.00390625f, 0.00390625f);
        const float2 h45 = __fmul2_rn(h01, k8), h67 = __fmul2_rn(h23, k8);
        acc[t][0] = __ffma2_rn(q[0], h01, acc[t][0]);
        acc[t][1] = __ffma2_rn(q[1], h23, acc[t][1]);
        acc[t][2] = __ffma2_rn(q[2], h45, acc[t][2]);
        acc[t][3] = __ffma2_rn(q[3], h67, acc[t][3]);
        acc[t][4] = __ffma2_rn(q[4], h01, acc[t][4]);
        acc[t][5] = __ffma2_rn(q[5], h23, acc[t][5]);
        acc[t][6] = __ffma2_rn(q[6], h45, acc[t][6]);
        acc[t][7] = __ffma2_rn(q[7], h67, acc[t][7]);
      }
    }
  }
}

// Sum over the 32 lanes of 16 values per lane; lane L receives the total of
// value index L >> 1 (lanes 2i and 2i+1 both hold total i).
__device__ __forceinline__ float reduce16(float (&v)[16]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int half = 8; half >= 1; half >>= 1) {
    const bool upper = (lane & (2 * half)) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float send = upper ? v[i] : v[i + half];
      const float keep = upper ? v[i + half] : v[i];
      v[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, 2 * half);
    }
  }
  return v[0] + __shfl_xor_sync(0xFFFFFFFFu, v[0], 1);
}

// Load the inputs of an item's tokens into shared memory, pre-scaled and
// laid out [token][float4 index q within a slice][slice s] (rows of NSL+1
// float4) so that the 32 lanes of a warp (consecutive slices) read
// consecutive 16-byte words; and the plain sum of each slice.  src(i) is the
// fp32 input of token i (n of them), NSL slices of 32 values.  Eight
// consecutive threads take the eight float4 of one slice (coalesced global
// reads, conflict-free stores thanks to the +1 row padding, slice sums by
// three shuffles); each thread keeps kStageUnroll loads in flight.
// Called by the nthreads consumer threads (a multiple of 32).
constexpr int kStageUnroll = 8;

template <int BITS, typename Src>
__device__ __forceinline__ void stage_inputs(float4* xs4, float* xsum, int n, int NSL, int nthreads, Src src) {
  const int per_tok = NSL * 8, total = n * per_tok, ld = NSL + 1;
  const int tid = threadIdx.x;
  for (int g0 = tid; g0 - tid < total; g0 += nthreads * kStageUnroll) {
    float4 v[kStageUnroll];
#pragma unroll
    for (int u = 0; u < kStageUnroll; ++u) {
      const int g = g0 + u * nthreads;
      if (g < total) {
        const int i = g / per_tok, rem = g - i * per_tok;
        v[u] = __ldcg(reinterpret_cast<const float4*>(src(i)) + rem);
      }
    }
#pragma unroll
    for (int u = 0; u < kStageUnroll; ++u) {
      const int g = g0 + u * nthreads;
      float sum = 0.f;
      if (g < total) {
        const int i = g / per_tok, rem = g - i * per_tok;
        const int s = rem >> 3, q = rem & 7;
        float4 w = v[u];
        sum = (w.x + w.y) + (w.z + w.w);
        w.x *= pos_scale<BITS>(4 * q + 0);
        w.y *= pos_scale<BITS>(4 * q + 1);
        w.z *= pos_scale<BITS>(4 * q + 2);
        w.w *= pos_scale<BITS>(4 * q + 3);
        xs4[(i * 8 + q) * ld + s] = w;
      }
      // groups of eight lanes hold one slice (total and nthreads are
      // multiples of 8, so a group is wholly in or out of range)
      sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 1);
      sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 2);
      sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 4);
      if (g < total && (g & 7) == 0) {
        const int i = g / per_tok, s = (g - i * per_tok) >> 3;
        xsum[i * NSL + s] = sum;
      }
    }
  }
}

// Bytes of shared memory that stage_inputs needs for G tokens of `cols` inputs.
static size_t staged_bytes(int cols, int G) {
  return (size_t)G * 8 * (cols / kSlice + 1) * 16 + (size_t)G * (cols / kSlice) * sizeof(float);
}

// Where the rows of a warp live: row r (0..3) has its codes at
// base + (r >> 1) * pair + (r & 1) * step and its (scale, bias) words at
// base + sb + (r >> 1) * pair + (r & 1) * sb_step.
struct RowAddr {
  uint32_t pair, step, sb, sb_step;
  __device__ __forceinline__ uint32_t q(int r) const { return (uint32_t)(r >> 1) * pair + (uint32_t)(r & 1) * step; }
  __device__ __forceinline__ uint32_t w(int r) const {
    return sb + (uint32_t)(r >> 1) * pair + (uint32_t)(r & 1) * sb_step;
  }
};

// acc[row][tok] = dot(row's codes, token tok's input) over the lane's slices,
// for the 4 rows at (base, ra) in shared memory and the NT tokens staged by
// stage_inputs.  Per slice the codes are masked once and meet every token
// from registers.
template <int BITS, int NT>
__device__ __forceinline__ void rows_dot(const uint8_t* base, const RowAddr ra, const float4* xs4,
                                         const float* xsum, int NSL, float (&acc)[4][kMaxTokGroup]) {
  const int lane = threadIdx.x & 31;
  const int ld = NSL + 1;
  for (int s = lane; s < NSL; s += 32) {
    SliceCodes<BITS> c[4];
    uint32_t sb[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      c[r] = smem_codes<BITS>(base + ra.q(r), s);
      sb[r] = reinterpret_cast<const uint32_t*>(base + ra.w(r))[s >> 1];
    }
    float2 pacc[4][NT];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int t = 0; t < NT; ++t) pacc[r][t] = make_float2(0.f, 0.f);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float2 xp[NT][4];
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        const float4 xa = xs4[(t * 8 + 2 * j) * ld + s];
        const float4 xb = xs4[(t * 8 + 2 * j + 1) * ld + s];
        xp[t][0] = make_float2(xa.x, xa.y);
        xp[t][1] = make_float2(xa.z, xa.w);
        xp[t][2] = make_float2(xb.x, xb.y);
        xp[t][3] = make_float2(xb.z, xb.w);
      }
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        float2 qp[4];
        octet_pairs(c[r], j, qp);
#pragma unroll
        for (int t = 0; t < NT; ++t)
#pragma unroll
          for (int i = 0; i < 4; ++i) pacc[r][t] = __ffma2_rn(qp[i], xp[t][i], pacc[r][t]);
      }
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const float s64 = bf16lo(sb[r]) * 18446744073709551616.0f;   // scale * 2^64
      const float b = bf16hi(sb[r]);
#pragma unroll
      for (int t = 0; t < NT; ++t) acc[r][t] += fmaf(s64, pacc[r][t].x + pacc[r][t].y, b * xsum[t * NSL + s]);
    }
  }
}

// rows_dot for the item's n tokens (1..4): the token count is a template
// argument so that no register or instruction is spent on absent tokens.
template <int BITS>
__device__ __forceinline__ void rows_dot_n(int n, const uint8_t* base, const RowAddr ra, const float4* xs4,
                                           const float* xsum, int NSL, float (&acc)[4][kMaxTokGroup]) {
  if (n == 1) rows_dot<BITS, 1>(base, ra, xs4, xsum, NSL, acc);
  else if (n == 2) rows_dot<BITS, 2>(base, ra, xs4, xsum, NSL, acc);
  else if (n == 3) rows_dot<BITS, 3>(base, ra, xs4, xsum, NSL, acc);
  else rows_dot<BITS, 4>(base, ra, xs4, xsum, NSL, acc);
}

__device__ __forceinline__ const uint8_t* item_blob(const BatchArgs& a, int expert) {
  return expert >= 0 ? a.experts + (size_t)expert * a.blob : a.shared;
}

// Shared control area of the expert kernels.
struct BatchCtrl {
  uint64_t full[kBatchMaxStages];
  uint64_t empty[kBatchMaxStages];
  uint64_t cbar;            // the consumer warps among themselves
  long long range[2];
  int item[kItemWords];
  int abort;
};
static_assert(sizeof(BatchCtrl) <= kBatchCtrlBytes, "control area");

// One work unit of an expert kernel: `rows` consecutive records of an
// expert, `rec_bytes` apart, starting at record `first` of the part that
// begins at byte `part` of the blob.
struct UnitShape {
  size_t part, rec_bytes;
  int rows;
};

constexpr int kCopiesPerUnit = 4;

// The producer side, run by the producer warp: stream the records of the
// block's units [u0, u1) into the ring, in order.  Lane 0 waits for free
// stages and declares each stage's bytes; the unit's copies are issued by
// lanes 0.. kCopiesPerUnit-1, one each: the copies one thread issues are
// carried out one after another, those of different threads side by side.
// Returns after the last copy has landed (bounded), so that no copy outlives
// the block.
__device__ void batch_produce(const BatchArgs& a, BatchCtrl* ctl, uint8_t* ring, int nstage, int stage_bytes,
                              long long u0, long long u1, int n_rb, const UnitShape us) {
  const int lane = threadIdx.x & 31;
  const uint32_t bytes = (uint32_t)(us.rows * us.rec_bytes);
  const int per = (us.rows + kCopiesPerUnit - 1) / kCopiesPerUnit;
  int cur_item = -1, expert = 0;
  long long k = 0;
  for (long long u = u0; u < u1; ++u, ++k) {
    const int st = (int)(k % nstage);
    const uint32_t use = (uint32_t)(k / nstage);
    bool ok = true;
    if (lane == 0 && use >= 1) ok = mbar_wait(&ctl->empty[st], (use - 1) & 1u, a.timeout_ns, a.err, &ctl->abort);
    if (!__shfl_sync(0xFFFFFFFFu, ok, 0)) break;
    const int item = (int)(u / n_rb), rb = (int)(u % n_rb);
    if (item != cur_item) {
      expert = __ldcg(a.plan + kPlanHeader + item * kItemWords);
      cur_item = item;
    }
    const uint8_t* src = item_blob(a, expert) + us.part + (size_t)rb * us.rows * us.rec_bytes;
    if (lane == 0) mbar_arrive_expect_tx(&ctl->full[st], bytes);
    __syncwarp();
    const int r0 = lane * per;
    if (lane < kCopiesPerUnit && r0 < us.rows) {
      const uint32_t b = (uint32_t)((us.rows - r0 < per ? us.rows - r0 : per) * us.rec_bytes);
      bulk_g2s(ring + (size_t)st * stage_bytes + (size_t)r0 * us.rec_bytes, src + (size_t)r0 * us.rec_bytes, b,
               &ctl->full[st]);
    }
  }
  // drain: every stage's last copy has landed before the block may exit
  if (lane == 0) {
    const long long issued = k;
    for (int st = 0; st < nstage && st < issued; ++st) {
      const long long last = st + ((issued - 1 - st) / nstage) * nstage;
      if (!mbar_wait_drain(&ctl->full[st], (uint32_t)(last / nstage) & 1u, a.timeout_ns)) {
        atomicOr(a.err, kErrCopyTimeout);
        ctl->abort = 1;
      }
    }
  }
  __syncwarp();
}

// Work units of this block: a contiguous share of the units (item-major,
// n_rb per item) holding an equal share of their total cost.  Called by every
// thread of the block (one thread per item looks for the two boundaries).
__device__ __forceinline__ void block_share(const BatchArgs& a, int n_rb, long long* range, long long& u0,
                                            long long& u1) {
  const int n_items = __ldcg(a.plan);
  const long long W = (long long)n_items * n_rb;
  const long long C = (long long)__ldcg(a.plan + 2) * n_rb;
  const long long x[2] = {C * blockIdx.x / gridDim.x, C * (blockIdx.x + 1) / gridDim.x};
  if (threadIdx.x == 0) range[0] = range[1] = W;
  __syncthreads();
  for (int i = threadIdx.x; i < n_items; i += blockDim.x) {
    const int32_t* it = a.plan + kPlanHeader + i * kItemWords;
    const long long c = unit_cost(__ldcg(it + 1));
    const long long q0 = (long long)__ldcg(it + 6) * n_rb, q1 = q0 + c * n_rb;
#pragma unroll
    for (int k = 0; k < 2; ++k)
      if (q0 <= x[k] && x[k] < q1) range[k] = (long long)i * n_rb + (x[k] - q0 + c - 1) / c;
  }
  __syncthreads();
  u0 = range[0];
  u1 = range[1];
}

__device__ __forceinline__ void batch_init(BatchCtrl* ctl, int nstage) {
  if (threadIdx.x == 0) {
    for (int i = 0; i < nstage; ++i) {
      mbar_init(&ctl->full[i], 1);
      mbar_init(&ctl->empty[i], kBatchConsumerWarps);
    }
    mbar_init(&ctl->cbar, kBatchConsumerWarps);
    ctl->abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
}

// ---------------------------------------------------------------------------
// gate/up + SwiGLU: unit = (item, gu_rows intermediate rows); consumer warp w
// < gu_warps takes records 2w and 2w+1 of the unit: gate and up of each
// ---------------------------------------------------------------------------
template <int BITS>
__global__ void __launch_bounds__(kBatchThreads, 1) batch_gateup_kernel(BatchArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  BatchCtrl* ctl = reinterpret_cast<BatchCtrl*>(smem);
  const BatchGeom& geo = a.geo;
  const int NSL = a.H / kSlice;
  float4* xs4 = reinterpret_cast<float4*>(smem + kBatchCtrlBytes);
  float* xsum = reinterpret_cast<float*>(xs4 + geo.G * 8 * (NSL + 1));
  uint8_t* ring = smem + kBatchCtrlBytes + geo.gu_xs_bytes;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int NS = a.K + a.S;
  const int n_rb = a.I / geo.gu_rows;
  long long u0, u1;
  block_share(a, n_rb, ctl->range, u0, u1);
  batch_init(ctl, geo.gu_nstage);

  if (warp == kBatchProducerWarp) {
    batch_produce(a, ctl, ring, geo.gu_nstage, geo.gu_stage_bytes, u0, u1, n_rb,
                  UnitShape{0, a.lay.gu_row, geo.gu_rows});
    return;
  }
  const RowAddr ra{(uint32_t)a.lay.gu_row, (uint32_t)a.lay.qh, (uint32_t)(2 * a.lay.qh), (uint32_t)a.lay.sh};
  // the consumer warps at one point: every warp arrives once per use, whole
  // (after __syncwarp); the wait is bounded
  uint32_t nsync = 0;
  auto cons_sync = [&]() -> bool {
    __syncwarp();
    if (lane == 0) mbar_arrive(&ctl->cbar);
    const bool ok = mbar_wait(&ctl->cbar, nsync & 1u, a.timeout_ns, a.err, &ctl->abort);
    ++nsync;
    return ok;
  };
  int cur = -1;
  long long k = 0;
  for (long long u = u0; u < u1; ++u, ++k) {
    const int item = (int)(u / n_rb), rb = (int)(u % n_rb);
    if (item != cur) {
      if (!cons_sync()) break;
      if (threadIdx.x < kItemWords) ctl->item[threadIdx.x] = __ldcg(a.plan + kPlanHeader + item * kItemWords + threadIdx.x);
      if (!cons_sync()) break;
      stage_inputs<BITS>(xs4, xsum, ctl->item[1], NSL, kBatchConsumerWarps * 32,
                         [&](int i) { return a.x + (size_t)(ctl->item[2 + i] >> 8) * a.H; });
      if (!cons_sync()) break;
      cur = item;
    }
    const int st = (int)(k % geo.gu_nstage);
    if (!mbar_wait(&ctl->full[st], (uint32_t)(k / geo.gu_nstage) & 1u, a.timeout_ns, a.err, &ctl->abort)) break;
    const int n = ctl->item[1];
    float acc[4][kMaxTokGroup] = {};
    if (warp < geo.gu_warps)
      rows_dot_n<BITS>(n, ring + (size_t)st * geo.gu_stage_bytes + (size_t)(2 * warp) * a.lay.gu_row, ra, xs4,
                       xsum, NSL, acc);
    __syncwarp();
    if (lane == 0) mbar_arrive(&ctl->empty[st]);
    if (warp < geo.gu_warps) {
      float v[16];
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int t = 0; t < kMaxTokGroup; ++t) v[r * kMaxTokGroup + t] = acc[r][t];
      const float tot = reduce16(v);
      // lane L holds value (row L >> 3, token (L >> 1) & 3); the up row of
      // the same token is 8 lanes up
      const float up = __shfl_xor_sync(0xFFFFFFFFu, tot, 8);
      const int tok = (lane >> 1) & 3;
      if ((lane & 9) == 0 && tok < n) {
        const int pr = ctl->item[2 + tok];
        const int r = rb * geo.gu_rows + 2 * warp + (lane >> 4);
        a.h[((size_t)(pr >> 8) * NS + (pr & 255)) * a.I + r] = silu_f(tot) * up;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// down: unit = (item, RB = 32*RW output rows).  The down projection is stored
// by column, so a unit needs a bx-byte slice (bx = 128, or the whole column
// when it is shorter) of each of the expert's I columns.  A 3-D tensor map
// over the pool (slice bytes x columns x experts) lets one tiled bulk copy
// fetch the slices of up to 256 consecutive columns into shared memory as a
// [column][bx] tile; the producer warp streams a unit's copies through a ring
// and consumer warp w takes columns [32w, 32w+32) of each tile: lane l the
// l-th code word of each column, i.e. rows r0 + l*RW .. r0 + l*RW + RW-1, for
// each of the item's tokens.  A warp's 32 columns lie in one 64-column group,
// whose scale and bias it applies at the end of the chunk; the eight warps'
// partial sums are added in a fixed order at the end of the unit.
// ---------------------------------------------------------------------------
struct BdCtrl {
  uint64_t full[kBdMaxStages];
  uint64_t empty[kBdMaxStages];
  uint64_t cbar;            // the consumer warps among themselves
  long long range[2];
  int item[kItemWords];
  int abort;
};
static_assert(sizeof(BdCtrl) <= kBdCtrlBytes, "control area");

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int x, int y, int z, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}

template <int BITS>
__global__ void __launch_bounds__(kBdThreads, 1) batch_down_kernel(BatchArgs a, float* __restrict__ y,
                                                                    const __grid_constant__ CUtensorMap tm_pool,
                                                                    const __grid_constant__ CUtensorMap tm_shared) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int RW = 32 / BITS;                    // rows per code word
  constexpr int RB = 32 * RW;                      // rows per unit
  constexpr int G = kMaxTokGroup;
  const BatchGeom& geo = a.geo;
  BdCtrl* ctl = reinterpret_cast<BdCtrl*>(smem);
  const int I = a.I, H = a.H, NS = a.K + a.S;
  const int bx = geo.bd_bx, box = geo.bd_box_cols;                            // tile: [box columns][bx bytes]
  float4* hsm = reinterpret_cast<float4*>(smem + kBdCtrlBytes);               // [G][I] h of the item's tokens, pre-scaled
  uint8_t* ring = smem + geo.bd_ring_off;                                     // [stage][box][bx]
  float* xbuf = reinterpret_cast<float*>(ring + (size_t)geo.bd_nstage * geo.bd_stage_bytes);   // [warp][RB][G]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_rb = (H + RB - 1) / RB;
  const int nc = (I + box - 1) / box;              // tiles per unit
  const int nst = geo.bd_nstage;                   // ring stages
  long long u0, u1;
  block_share(a, n_rb, ctl->range, u0, u1);
  if (tid == 0) {
    for (int i = 0; i < nst; ++i) {
      mbar_init(&ctl->full[i], 1);
      mbar_init(&ctl->empty[i], kBdWarps);
    }
    mbar_init(&ctl->cbar, kBdWarps);
    ctl->abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  volatile int* abort = &ctl->abort;
  const uint32_t tile_bytes = (uint32_t)(box * bx);

  if (warp == kBdWarps) {
    // ---- producer: lane 0 issues every tile of the block's units, in order
    long long k = 0;
    if (lane == 0) {
      int cur = -1, expert = 0;
      for (long long u = u0; u < u1 && !*abort; ++u) {
        const int item = (int)(u / n_rb), rb = (int)(u % n_rb);
        if (item != cur) {
          expert = __ldcg(a.plan + kPlanHeader + item * kItemWords);
          cur = item;
        }
        const CUtensorMap* map = expert >= 0 ? &tm_pool : &tm_shared;
        const int z = expert >= 0 ? expert : 0;
        const int x = rb * RB * BITS / 8;          // a multiple of 128 bytes
        for (int c = 0; c < nc; ++c, ++k) {
          const int st = (int)(k % nst);
          const uint32_t use = (uint32_t)(k / nst);
          if (use >= 1 && !mbar_wait(&ctl->empty[st], (use - 1) & 1u, a.timeout_ns, a.err, abort)) break;
          mbar_arrive_expect_tx(&ctl->full[st], tile_bytes);
          tma_load_3d(ring + (size_t)st * geo.bd_stage_bytes, map, x, c * box, z, &ctl->full[st]);
        }
      }
      // drain: every stage's last copy has landed before the block may exit
      for (int st = 0; st < nst && st < k; ++st) {
        const long long last = st + ((k - 1 - st) / nst) * nst;
        if (!mbar_wait_drain(&ctl->full[st], (uint32_t)(last / nst) & 1u, a.timeout_ns)) {
          atomicOr(a.err, kErrCopyTimeout);
          ctl->abort = 1;
        }
      }
    }
    __syncwarp();
    return;
  }

  // ---- consumers
  uint32_t nsync = 0;
  // the eight consumer warps at one point (bounded)
  auto cons_sync = [&]() -> bool {
    __syncwarp();
    if (lane == 0) mbar_arrive(&ctl->cbar);
    const bool ok = mbar_wait(&ctl->cbar, nsync & 1u, a.timeout_ns, a.err, abort);
    ++nsync;
    return ok;
  };
  long long k = 0;
  int cur = -1;
  for (long long u = u0; u < u1; ++u) {
    const int item = (int)(u / n_rb), rb = (int)(u % n_rb);
    const int r0 = rb * RB;
    if (item != cur) {
      if (!cons_sync()) break;                     // every warp is done with the previous item
      if (tid < kItemWords) ctl->item[tid] = __ldcg(a.plan + kPlanHeader + item * kItemWords + tid);
      if (!cons_sync()) break;
      const int n = ctl->item[1];
      for (int idx = tid; idx < n * I; idx += kBdWarps * 32) {
        const int t = idx / I, i = idx - t * I;
        const int pr = ctl->item[2 + t];
        const float hv = __ldcg(a.h + ((size_t)(pr >> 8) * NS + (pr & 255)) * I + i);
        hsm[t * I + i] = make_float4(hv * pos_scale<BITS>(0), hv * pos_scale<BITS>(1), hv * pos_scale<BITS>(2),
                                     hv * pos_scale<BITS>(3));
      }
      if (!cons_sync()) break;
      cur = item;
    }
    const int n = ctl->item[1];
    const uint8_t* blob = item_blob(a, ctl->item[0]);
    const int vb = min(bx, (H - r0) * BITS / 8);      // valid bytes of a column's slice (a multiple of 16)
    const bool row_ok = lane * 4 < vb;

    float outp[RW][G];
#pragma unroll
    for (int r = 0; r < RW; ++r)
#pragma unroll
      for (int t = 0; t < G; ++t) outp[r][t] = 0.f;
    for (int c = 0; c < nc; ++c, ++k) {
      const int st = (int)(k % nst);
      const bool ok = mbar_wait(&ctl->full[st], (uint32_t)(k / nst) & 1u, a.timeout_ns, a.err, abort);
      const int col0 = c * box + 32 * warp;            // this warp's first column of the tile
      if (ok && 32 * warp < box && col0 < I) {
        // the group's (scale, bias) words of the lane's rows
        uint32_t sbv[RW];
        {
          const uint4* src = reinterpret_cast<const uint4*>(blob + a.lay.dsb_off + (size_t)(col0 / kGroup) * a.lay.dsb_group +
                                                            (size_t)(r0 + RW * lane) * 4);
#pragma unroll
          for (int q = 0; q < RW / 4; ++q) {
            const uint4 v = row_ok ? __ldg(src + q) : make_uint4(0u, 0u, 0u, 0u);
            sbv[4 * q] = v.x; sbv[4 * q + 1] = v.y; sbv[4 * q + 2] = v.z; sbv[4 * q + 3] = v.w;
          }
        }
        float2 acc[G][RW / 2];
        float hs[G];
#pragma unroll
        for (int t = 0; t < G; ++t) {
          hs[t] = 0.f;
#pragma unroll
          for (int r = 0; r < RW / 2; ++r) acc[t][r] = make_float2(0.f, 0.f);
        }
        const uint8_t* tile = ring + (size_t)st * geo.bd_stage_bytes + (size_t)(32 * warp) * bx;
        const int ncol = min(32, I - col0);
        const float4* hq = hsm + col0;
        if (n == 1) bd_columns<BITS, 1>(tile, bx, ncol, row_ok, hq, I, acc, hs);
        else if (n == 2) bd_columns<BITS, 2>(tile, bx, ncol, row_ok, hq, I, acc, hs);
        else if (n == 3) bd_columns<BITS, 3>(tile, bx, ncol, row_ok, hq, I, acc, hs);
        else bd_columns<BITS, 4>(tile, bx, ncol, row_ok, hq, I, acc, hs);
#pragma unroll
        for (int t = 0; t < G; ++t) hs[t] *= inv_pos_scale<BITS>(0);   // exact: a power of two
        // out += s * 2^64 * acc + b * sum(h) over the chunk's columns
#pragma unroll
        for (int t = 0; t < G; ++t) {
#pragma unroll
          for (int r = 0; r < RW / 2; ++r) {
            outp[2 * r][t] += fmaf(bf16lo(sbv[2 * r]) * 18446744073709551616.0f, acc[t][r].x, bf16hi(sbv[2 * r]) * hs[t]);
            outp[2 * r + 1][t] +=
                fmaf(bf16lo(sbv[2 * r + 1]) * 18446744073709551616.0f, acc[t][r].y, bf16hi(sbv[2 * r + 1]) * hs[t]);
          }
        }
      }
      // the tile may be refilled
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->empty[st]);
    }
    // the eight warps' partial sums, added in warp order; a warp's buffer is
    // [row within the lane's word][token][lane], so that both the writes and
    // the reads below touch 32 consecutive words (no bank conflicts)
    float* xb = xbuf + (size_t)warp * RB * G;
#pragma unroll
    for (int r = 0; r < RW; ++r)
#pragma unroll
      for (int t = 0; t < G; ++t) xb[(r * G + t) * 32 + lane] = outp[r][t];
    if (!cons_sync()) break;
    for (int idx = tid; idx < RB * n; idx += kBdWarps * 32) {
      const int ln = idx & 31, rest = idx >> 5;
      const int r = rest % RW, t = rest / RW;
      const int row = RW * ln + r;
      if (r0 + row < H) {
        float v = 0.f;
#pragma unroll
        for (int w2 = 0; w2 < kBdWarps; ++w2) v += xbuf[(size_t)w2 * RB * G + (r * G + t) * 32 + ln];
        const int pr = ctl->item[2 + t];
        y[((size_t)(pr >> 8) * NS + (pr & 255)) * H + r0 + row] = v;
      }
    }
    if (!cons_sync()) break;
  }
}

// out[t] = residual[t] + sum_k w[t][k] y[t][k] + g[t] y[t][K]
__global__ void batch_combine_kernel(BatchArgs a) {
  const int H4 = a.H / 4;
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= a.T * H4) return;
  const int t = idx / H4, j4 = idx % H4;
  const int NS = a.K + a.S;
  const float4* y4 = reinterpret_cast<const float4*>(a.y);
  float4 acc = reinterpret_cast<const float4*>(a.residual)[idx];
  auto add = [&](float w, int slot) {
    const float4 v = y4[((size_t)t * NS + slot) * H4 + j4];
    acc.x = fmaf(w, v.x, acc.x);
    acc.y = fmaf(w, v.y, acc.y);
    acc.z = fmaf(w, v.z, acc.z);
    acc.w = fmaf(w, v.w, acc.w);
  };
  for (int k = 0; k < a.K; ++k) add(a.weights[t * a.K + k], k);
  if (a.S) add(a.gate[t], a.K);
  reinterpret_cast<float4*>(a.out)[idx] = acc;
}

// x = h / sqrt(mean(h^2) + eps) (unit weight), one token: the general path
// of a stack (the persistent kernel normalises in its own input phase)
cudaError_t launch_rmsnorm(const float* h, float* x, int H, float eps, cudaStream_t st) {
  return launch_rmsnorm_w(h, nullptr, 1, H, eps, x, st);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
cudaError_t launch_route(const float* logits, int T, int E, int K, int32_t* ids, float* weights,
                         const uint16_t* wsg, const float* x, int H, float* gate, cudaStream_t st) {
  const int warps = 4;
  route_kernel<<<(T + warps - 1) / warps, 32 * warps, 0, st>>>(logits, T, E, K, ids, weights, wsg, x,
                                                                 H, gate);
  return cudaGetLastError();
}

int batch_max_items(int T, int K, int S, int G) { return T * K + S * ((T + G - 1) / G); }

static size_t round_up128(size_t v) { return (v + 127) / 128 * 128; }

BatchGeom batch_geometry(int bits, int H, int I, int device) {
  int sms = 0, smem_max = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess ||
      cudaDeviceGetAttribute(&smem_max, cudaDevAttrMaxSharedMemoryPerBlockOptin, device) != cudaSuccess) {
    cudaGetLastError();
    return BatchGeom{};
  }
  return batch_geometry_for(bits, H, I, sms, smem_max);
}

BatchGeom batch_geometry_for(int bits, int H, int I, int sms, int smem_max) {
  BatchGeom g{};
  if (sms < 1 || smem_max <= kBatchCtrlBytes) return g;
  const BlobLayout lay = blob_layout(bits, H, I);
  const size_t avail = (size_t)smem_max - kBatchCtrlBytes;
  const int rb = 32 * (32 / bits);                  // output rows per down unit
  // a down tile: up to 256 columns' 128-byte slices (the whole column when
  // it is shorter); stages 1 KB aligned
  const int bx = (int)std::min<size_t>(128, lay.dcol);
  const int box = std::min(kBdMaxBoxCols, I);
  const size_t bd_stage = (size_t)box * bx;
  // the most tokens per item, then the most gate/up warps, for which two
  // gate/up ring stages fit next to the staged inputs, and the down kernel's
  // staged h, ring and partial sums fit
  for (int G = kMaxTokGroup; G >= 1; G /= 2) {
    const size_t gx = round_up128(staged_bytes(H, G));
    // h staged pre-scaled (a float4 per token and column); as many ring
    // stages as fit, at least two
    const size_t bdh = round_up128((size_t)G * I * 16);
    const size_t ring_off = (kBdCtrlBytes + bdh + 1023) / 1024 * 1024;
    const size_t xb = (size_t)kBdWarps * rb * kMaxTokGroup * 4;
    if (ring_off + 2 * bd_stage + xb > (size_t)smem_max) continue;
    const int bd_nst = (int)std::min<size_t>(kBdMaxStages, ((size_t)smem_max - ring_off - xb) / bd_stage);
    const size_t bd_smem = ring_off + (size_t)bd_nst * bd_stage + xb;
    for (int w = kBatchConsumerWarps; w >= 1; w /= 2) {
      const size_t gu_stage = round_up128((size_t)2 * w * lay.gu_row);
      if (I % (2 * w) || gx + 2 * gu_stage > avail) continue;
      g.G = G;
      g.gu_warps = w;
      g.gu_rows = 2 * w;
      g.gu_stage_bytes = (int)gu_stage;
      g.gu_nstage = (int)std::min<size_t>(kBatchMaxStages, (avail - gx) / gu_stage);
      g.gu_xs_bytes = (int)gx;
      g.gu_smem = kBatchCtrlBytes + gx + (size_t)g.gu_nstage * gu_stage;
      g.bd_h_bytes = (int)bdh;
      g.bd_bx = bx;
      g.bd_box_cols = box;
      g.bd_stage_bytes = (int)bd_stage;
      g.bd_ring_off = (int)ring_off;
      g.bd_nstage = bd_nst;
      g.bd_smem = bd_smem;
      g.grid = sms;
      return g;
    }
  }
  return g;
}

// Raise a kernel's dynamic shared-memory limit to `bytes` (once per kernel,
// device and size; `done` remembers the largest size set so far).
template <typename Kern>
static cudaError_t allow_smem(Kern k, size_t bytes, size_t& done) {
  if (bytes <= 48 * 1024 || bytes <= done) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess) done = bytes;
  return e;
}
// per device: gate/up 4-bit, 2-bit; down 4-bit, 2-bit (function attributes
// belong to the device's context)
static size_t g_smem_set[64][4];
static std::mutex g_smem_mu;

// cuTensorMapEncodeTiled (a CUDA driver API entry point), looked up once
// through the runtime, so that the library need not link libcuda.
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    else
      cudaGetLastError();
  });
  return fn;
}

// Tensor map over the down codes of `n` blobs `blob` bytes apart from
// `base`: dimensions (slice bytes, columns, blobs), tile [box columns][bx].
static bool down_tensor_map(CUtensorMap* m, const uint8_t* base, int n, const BatchArgs& a) {
  const PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)a.lay.dcol, (cuuint64_t)a.I, (cuuint64_t)n};
  const cuuint64_t strides[2] = {(cuuint64_t)a.lay.dcol, (cuuint64_t)a.blob};
  const cuuint32_t box[3] = {(cuuint32_t)a.geo.bd_bx, (cuuint32_t)a.geo.bd_box_cols, 1u};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t*>(base + a.lay.dq_off), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_batch(BatchArgs& a, float* y, cudaStream_t st) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  a.geo = batch_geometry(a.bits, a.H, a.I, dev);
  if (a.geo.grid == 0) return cudaErrorInvalidValue;
  size_t* set = g_smem_set[dev];
  std::lock_guard<std::mutex> lock(g_smem_mu);

  batch_plan_kernel<<<1, kPlanThreads, 0, st>>>(a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;

  const BatchGeom& g = a.geo;
  if (a.bits == 4) {
    if ((e = allow_smem(batch_gateup_kernel<4>, g.gu_smem, set[0])) != cudaSuccess) return e;
    batch_gateup_kernel<4><<<g.grid, kBatchThreads, g.gu_smem, st>>>(a);
  } else {
    if ((e = allow_smem(batch_gateup_kernel<2>, g.gu_smem, set[1])) != cudaSuccess) return e;
    batch_gateup_kernel<2><<<g.grid, kBatchThreads, g.gu_smem, st>>>(a);
  }
  if ((e = cudaGetLastError()) != cudaSuccess) return e;

  CUtensorMap tm_pool, tm_shared;
  if (!down_tensor_map(&tm_pool, a.experts, a.E, a) ||
      !down_tensor_map(&tm_shared, a.S ? a.shared : a.experts, 1, a))
    return cudaErrorInvalidValue;
  if (a.bits == 4) {
    if ((e = allow_smem(batch_down_kernel<4>, g.bd_smem, set[2])) != cudaSuccess) return e;
    batch_down_kernel<4><<<g.grid, kBdThreads, g.bd_smem, st>>>(a, y, tm_pool, tm_shared);
  } else {
    if ((e = allow_smem(batch_down_kernel<2>, g.bd_smem, set[3])) != cudaSuccess) return e;
    batch_down_kernel<2><<<g.grid, kBdThreads, g.bd_smem, st>>>(a, y, tm_pool, tm_shared);
  }
  if ((e = cudaGetLastError()) != cudaSuccess) return e;

  if (a.out != nullptr) {
    const int n = a.T * (a.H / 4);
    batch_combine_kernel<<<(n + 255) / 256, 256, 0, st>>>(a);
    e = cudaGetLastError();
  }
  return e;
}

}  // namespace fmoe
