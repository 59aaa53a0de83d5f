// Kernel argument structs and launcher declarations shared by the .cu files.
#pragma once

#include "fmoe_internal.cuh"

namespace fmoe {

// Geometry of the batched expert kernels (host computed by batch_geometry).
struct BatchGeom {
  int G;                    // tokens per plan item (4, 2 or 1: what the staged inputs leave room for)
  int gu_warps;             // consumer warps with gate/up rows (2 rows each per unit)
  int gu_rows;              // intermediate rows per gate/up work unit (2 * gu_warps)
  int gu_nstage, gu_stage_bytes;
  int gu_xs_bytes;                // staged inputs
  int bd_h_bytes;                 // down: staged h of an item's tokens
  int bd_bx, bd_box_cols;         // down: tile of a tensor copy, [bd_box_cols columns][bd_bx bytes]
  int bd_stage_bytes, bd_ring_off, bd_nstage;
  size_t gu_smem, bd_smem;
  int grid;
};

// Arguments of the routing and batched kernels (fmoe_batch.cu).
struct BatchArgs {
  int bits, H, I, E, K, S, T;
  size_t blob;
  BlobLayout lay;
  const uint8_t* experts;
  const uint8_t* shared;
  const float* logits;      // [T][E]: route in the plan kernel; nullptr: ids_in given
  const int32_t* ids_in;    // [T][K] caller's ids (fmoe_expert_ffn) or nullptr
  const uint16_t* wsg;      // shared gate vector [H] (S == 1, routing) or nullptr
  int32_t* ids;             // [T][K] routing result
  float* weights;           // [T][K]
  float* gate;              // [T]
  const float* x;           // [T][H]
  const float* residual;    // [T][H]
  float* out;               // [T][H], or nullptr: stop after y
  float* h;                 // [T][K+S][I]
  float* y;                 // [T][K+S][H] unweighted expert outputs
  int32_t* plan;            // batch plan (fmoe_batch.cu)
  uint32_t* err;
  unsigned long long timeout_ns;
  BatchGeom geo;
};

constexpr int kMaxTokGroup = 4;        // most tokens that share one pass over an expert's codes
constexpr int kPlanHeader = 8;         // int32: [0] items, [1] distinct experts (incl. shared)
constexpr int kItemWords = 8;          // int32 per plan item
constexpr int kBatchConsumerWarps = 8;
constexpr int kBatchProducerWarp = kBatchConsumerWarps;
constexpr int kBatchThreads = 32 * (kBatchConsumerWarps + 1);
constexpr int kBatchMaxStages = 8;
// down kernel: consumer warps (32 columns of each tile each), one producer
// warp, ring stages of one tensor tile, most columns per tile
constexpr int kBdWarps = 8;
constexpr int kBdThreads = 32 * (kBdWarps + 1);
constexpr int kBdMaxStages = 4;
constexpr int kBdMaxBoxCols = 32 * kBdWarps;
constexpr int kBdCtrlBytes = 256;
constexpr int kBatchCtrlBytes = 256;   // mbarriers, work range, item header at the start of shared memory

// Largest number of plan items for T tokens, top-K, S shared experts, G
// tokens per item.
int batch_max_items(int T, int K, int S, int G);
// Geometry for a shape; grid == 0 if it does not fit (never for the shapes
// the ABI accepts).
BatchGeom batch_geometry(int bits, int H, int I, int device);
// The same for a device with `sms` SMs and `smem_max` bytes of shared memory
// per block (host arithmetic only).
BatchGeom batch_geometry_for(int bits, int H, int I, int sms, int smem_max);

// RMSNorm block size (fmoe_dense.cu)
constexpr int kNormThreads = 1024;
// record bytes of a dense quantised row; y[t] = W x[t] (+ residual[t]) for
// a dense matrix of N row records; x = RMSNorm(h) (* w) for T tokens
// (fmoe_dense.cu)
int dense_row_bytes(int bits, int H);
cudaError_t launch_dense_gemv(const uint8_t* w, int bits, int N, int H, const float* x, int T, const float* residual,
                              float* y, cudaStream_t st);
cudaError_t launch_rmsnorm_w(const float* h, const float* w, int T, int H, float eps, float* x, cudaStream_t st);
// logits[t][e] = w[e] . x[t] (fmoe_router.cu)
cudaError_t launch_router(const uint16_t* w, const float* x, int T, int H, int E, float* logits, cudaStream_t st);
cudaError_t launch_route(const float* logits, int T, int E, int K, int32_t* ids, float* weights,
                         const uint16_t* wsg, const float* x, int H, float* gate, cudaStream_t st);
// plan -> gate/up -> down into y (-> combine into a.out when non-null)
cudaError_t launch_batch(BatchArgs& a, float* y, cudaStream_t st);
// x = h / sqrt(mean(h^2) + eps)
cudaError_t launch_rmsnorm(const float* h, float* x, int H, float eps, cudaStream_t st);

// ---------------------------------------------------------------------------
// single-launch persistent kernel (fmoe_fused.cu)
// ---------------------------------------------------------------------------
constexpr int kGuWarps = 12;                           // dequantised gate/up GEMV warps
constexpr int kDnWarps = 8;                            // down projection warps
constexpr int kPollWarps = kGuWarps + kDnWarps;        // warps that gather each layer's input
constexpr int kProducerWarp = kPollWarps;              // issues the bulk copies
constexpr int kFinalWarp = kPollWarps + 1;             // routes, turns partial sums into h
constexpr int kFusedWarps = kPollWarps + 2;
constexpr int kFusedThreads = 32 * kFusedWarps;
constexpr int kDnThreads = 32 * kDnWarps;
// registers per thread: the SM's 64K registers shared by the block's threads
constexpr int kFusedMaxRegs = (65536 / kFusedThreads) / 8 * 8;
constexpr int kMaxFusedLayers = 64;    // layers per launch; longer stacks use several launches
constexpr int kMaxSlots = FMOE_MAX_TOPK + 1;
constexpr int kMaxStages = 16;
constexpr int kMaxPieces = 4;          // slot ranges a block's columns may span
constexpr int kCtrlBytes = 2048;       // barriers, pieces, routing result, reductions
// Tuning of the persistent kernel (compile-time; the defaults are the
// measured best): ring stages at most, ring stages issued before a layer's
// down columns, most bytes per bulk copy (the TMA unit spends about half a
// microsecond per copy whatever its size, so a block streams fastest with
// few large copies: 16 KB copies cap an SM near 33 GB/s, 32 KB and larger
// near 47 GB/s), producer lanes that take turns issuing copies, pause
// between two polls of the accumulators.
#ifndef FMOE_FUSED_STAGE_CAP
#define FMOE_FUSED_STAGE_CAP 8
#endif
#ifndef FMOE_FUSED_DAREA_AFTER
#define FMOE_FUSED_DAREA_AFTER 2
#endif
#ifndef FMOE_FUSED_COPY_BYTES
#define FMOE_FUSED_COPY_BYTES (1u << 19)
#endif
#ifndef FMOE_FUSED_ISSUE_LANES
#define FMOE_FUSED_ISSUE_LANES 4
#endif
#ifndef FMOE_POLL_NS
#define FMOE_POLL_NS 64
#endif
#ifndef FMOE_WAIT_NS
#define FMOE_WAIT_NS 32
#endif
#ifndef FMOE_FINAL_SPIN
#define FMOE_FINAL_SPIN 0
#endif
#ifndef FMOE_FUSED_SB_GLOBAL
#define FMOE_FUSED_SB_GLOBAL 0
#endif
#ifndef FMOE_FUSED_SHARED_WEIGHT
#define FMOE_FUSED_SHARED_WEIGHT 100
#endif

constexpr int kFusedStageCap = FMOE_FUSED_STAGE_CAP < kMaxStages ? FMOE_FUSED_STAGE_CAP : kMaxStages;
constexpr int kFusedDareaAfter = FMOE_FUSED_DAREA_AFTER;
constexpr uint32_t kFusedCopyBytes = FMOE_FUSED_COPY_BYTES;
constexpr int kFusedIssueLanes = FMOE_FUSED_ISSUE_LANES;
constexpr unsigned kPollNs = FMOE_POLL_NS;
// 1: the down groups' (scale,bias) words are read from L2 at each group's
// fold (asked into L2 when the layer starts) instead of being copied into
// shared memory, and the ring gets the space (4 stages instead of 3 at the
// Qwen shape); measured 1 % slower, so off
constexpr bool kFusedSbGlobal = FMOE_FUSED_SB_GLOBAL != 0;
// pause between two checks of a counter the down warps wait on (0: spin):
// spinning warps take issue slots and shared-memory bandwidth from the
// gate/up warps, which set the pace of the ring (32 ns measured 1 % faster
// than spinning at the Qwen 4-bit shape)
constexpr unsigned kWaitNs = FMOE_WAIT_NS;
// 1: the finaliser spins on the gate/up warps' partial sums; 0: it waits
// suspended in the barrier unit (measured no slower, and it frees issue slots)
constexpr bool kFinalSpin = FMOE_FINAL_SPIN != 0;
// cost of a shared-expert column against a routed one, in percent, when the
// blocks' columns are split: the shared expert needs no routing and is
// streamed during the previous layer's exchange, so a lower cost gives its
// blocks more columns and every routed block fewer
constexpr int kFusedSharedWeight = FMOE_FUSED_SHARED_WEIGHT;

// A block's intermediate columns within one slot: columns [i0, i0+cnt) of
// slot `slot`, local indices [loc, loc+cnt); in the block's down area its
// columns' codes at col_off and the (scale,bias) words of groups g0..g0+ng-1
// at sb_off.
struct Piece {
  int slot, i0, cnt, loc, col_off, sb_off, g0, ng;
};

// The virtual columns [v0, v1) of block c of n in the slot-major sequence
// (slot 0 = the shared expert when S = 1): equal shares of the total cost,
// a shared column costing kFusedSharedWeight percent of a routed one.
__host__ __device__ inline void block_bounds(int NS, int I, int S, int c, int n, long long& v0, long long& v1) {
  const long long ws = S ? kFusedSharedWeight : 100;
  const long long cs = (long long)S * I * ws;                       // cost of the shared columns
  const long long C = cs + (long long)(NS - S) * I * 100;
  auto col = [&](long long x) -> long long { return x <= cs ? x / ws : (long long)S * I + (x - cs) / 100; };
  v0 = col(C * c / n);
  v1 = col(C * (c + 1) / n);
}

// Columns of block c of n (block_bounds), split at slot boundaries.  Returns
// the number of pieces (at most max_pieces are written) and the down-area
// bytes they need.
__host__ __device__ inline int block_pieces(int NS, int I, int S, int c, int n, const BlobLayout& lay, Piece* pc,
                                            int max_pieces, int& darea_bytes) {
  long long v, v1;
  block_bounds(NS, I, S, c, n, v, v1);
  int np = 0, off = 0, u = 0;
  while (v < v1) {
    const int slot = (int)(v / I), i0 = (int)(v % I);
    const int cnt = (int)((v1 - v) < (long long)(I - i0) ? (v1 - v) : (long long)(I - i0));
    const int g0 = i0 / kGroup, ng = (i0 + cnt - 1) / kGroup - g0 + 1;
    const int cb = (int)round_up((size_t)cnt * lay.dcol, 128), sbb = (int)round_up((size_t)ng * lay.dsb_group, 128);
    if (np < max_pieces) pc[np] = Piece{slot, i0, cnt, u, off, off + cb, g0, ng};
    off += cb + (kFusedSbGlobal ? 0 : sbb);
    u += cnt;
    v += cnt;
    ++np;
  }
  darea_bytes = off;
  return np;
}

struct FusedLayerPtrs {
  const uint8_t* experts;
  const uint8_t* shared;
  const uint16_t* wsg;
};

// Shared-memory plan and per-shape geometry (host computed by fused_plan).
struct FusedPlan {
  bool ok;
  int grid;
  size_t smem;
  int R;                    // gate/up records per ring stage (two per gate/up warp and slice range)
  int nparts;               // partial sums per gate/up row (slice ranges of H)
  int nstage, stage_bytes;  // ring
  int len_max;              // most intermediate columns a block owns
  int hb;                   // floats per column in the h buffer
  int xs_off, part_off, hbuf_off, dscr_off, darea_off, darea_bytes, ring_off;
};

struct FusedParams {
  int bits, H, I, E, K, S, L;
  int norm;                 // 1: input = RMSNorm(h), residual = h (stack); 0: given x / residual
  float eps;
  size_t blob;
  BlobLayout lay;
  const float* x;           // norm == 0: input [H]
  const float* residual;    // norm == 0: residual [H]
  float* out;               // norm == 0: output [H];  norm == 1: h (in for layer 0, out after the last)
  const float* logits;      // [L][E]
  float* hmid;              // [K+S][I] h of the last layer (plain fp32), or nullptr
  unsigned long long* acc;  // [3][H] fixed-point accumulators (workspace state)
  uint32_t* lbase;          // layers run on the workspace, modulo 3
  int32_t* ids_out;         // [L][K] or nullptr
  float* w_out;             // [L][K] or nullptr
  float* gate_out;          // [L] or nullptr
  uint32_t* exit_ctr;       // zero on entry and on exit
  uint32_t* err;
  unsigned long long timeout_ns;
  FusedPlan plan;
  FusedLayerPtrs layer[kMaxFusedLayers];
};

// Plan the persistent launch for a shape; ok == false if the shape does not
// fit the kernel's limits (the caller then uses the general kernels).
FusedPlan fused_plan(int bits, int H, int I, int K, int S, int device);
// The same for a device with `sms` SMs and `smem_max` bytes of shared memory
// per block (host arithmetic only).
FusedPlan fused_plan_for(int bits, int H, int I, int K, int S, int sms, int smem_max);
cudaError_t launch_fused(FusedParams& p, const FusedPlan& plan, cudaStream_t st);

// ---------------------------------------------------------------------------
// host-side argument checks shared by the entry points
// ---------------------------------------------------------------------------
inline bool host_aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

inline bool host_vec_ok(const void* p) { return p != nullptr && host_aligned(p, 16); }

inline bool host_overlap(const void* a, size_t na, const void* b, size_t nb) {
  const char* pa = static_cast<const char*>(a);
  const char* pb = static_cast<const char*>(b);
  return pa < pb + nb && pb < pa + na;
}

// Shape and pointer checks common to every call that reads expert blobs.
inline fmoe_status check_layer(const fmoe_layer* L, bool need_ptrs) {
  if (L == nullptr) return FMOE_ERR_INVALID_ARG;
  if (L->bits != 4 && L->bits != 2) return FMOE_ERR_UNSUPPORTED;
  if (L->group != kGroup) return FMOE_ERR_UNSUPPORTED;
  if (L->hidden <= 0 || L->inter <= 0 || L->hidden % kGroup || L->inter % kGroup) return FMOE_ERR_INVALID_ARG;
  if (L->hidden > FMOE_MAX_HIDDEN || L->inter > FMOE_MAX_INTER) return FMOE_ERR_UNSUPPORTED;
  if (L->n_experts <= 0 || L->n_experts > FMOE_MAX_EXPERTS) return FMOE_ERR_INVALID_ARG;
  if (L->has_shared != 0 && L->has_shared != 1) return FMOE_ERR_INVALID_ARG;
  if (need_ptrs) {
    if (L->experts == nullptr || !host_aligned(L->experts, kPlaneAlign)) return FMOE_ERR_INVALID_ARG;
    if (L->has_shared) {
      if (L->shared == nullptr || !host_aligned(L->shared, kPlaneAlign)) return FMOE_ERR_INVALID_ARG;
      if (L->shared_gate_w == nullptr || !host_aligned(L->shared_gate_w, 16)) return FMOE_ERR_INVALID_ARG;
    }
  }
  return FMOE_OK;
}

// The activation arguments of fmoe_moe_block (T tokens): non-null, 16-byte
// aligned; out may alias residual but must not overlap x or the logits.
inline fmoe_status check_block_args(const fmoe_layer* L, const float* x, const float* logits,
                                    const float* residual, const float* out, int T) {
  if (!host_vec_ok(x) || !host_vec_ok(logits) || !host_vec_ok(residual) || !host_vec_ok(out))
    return FMOE_ERR_INVALID_ARG;
  const size_t hb = (size_t)T * L->hidden * 4;
  if (host_overlap(out, hb, x, hb) || host_overlap(out, hb, logits, (size_t)T * L->n_experts * 4))
    return FMOE_ERR_INVALID_ARG;
  if (out != residual && host_overlap(out, hb, residual, hb)) return FMOE_ERR_INVALID_ARG;
  return FMOE_OK;
}

// Fill the persistent kernel's per-call fields for layer descriptors
// layers[0..n) (same shape), n <= kMaxFusedLayers.
inline void fused_params_for(FusedParams& p, const fmoe_layer* layers, int n, int K) {
  const fmoe_layer& L0 = layers[0];
  p.bits = L0.bits;
  p.H = L0.hidden;
  p.I = L0.inter;
  p.E = L0.n_experts;
  p.K = K;
  p.S = L0.has_shared;
  p.L = n;
  p.lay = blob_layout(L0.bits, L0.hidden, L0.inter);
  p.blob = p.lay.bytes;
  for (int i = 0; i < n; ++i) {
    p.layer[i].experts = static_cast<const uint8_t*>(layers[i].experts);
    p.layer[i].shared = static_cast<const uint8_t*>(layers[i].shared);
    p.layer[i].wsg = layers[i].shared_gate_w;
  }
}

cudaError_t launch_wait_test(uint32_t* counter, uint32_t* err, int n_blocks, int expected,
                             unsigned long long timeout_ns, cudaStream_t st);

}  // namespace fmoe
