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
  int d_nstage, d_stage_bytes;    // down: 4 rows per consumer warp per unit
  int gu_xs_bytes, d_xs_bytes;    // staged inputs
  size_t gu_smem, d_smem;
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
constexpr int kDownRowsPerWarp = 4;
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

cudaError_t launch_route(const float* logits, int T, int E, int K, int32_t* ids, float* weights,
                         const uint16_t* wsg, const float* x, int H, float* gate, cudaStream_t st);
// plan -> gate/up -> down into y (-> combine into a.out when non-null)
cudaError_t launch_batch(BatchArgs& a, float* y, cudaStream_t st);

// ---------------------------------------------------------------------------
// single-launch persistent kernel (fmoe_fused.cu)
// ---------------------------------------------------------------------------
#ifndef FMOE_FUSED_GU_WARPS
#define FMOE_FUSED_GU_WARPS 12
#endif
constexpr int kGuWarps = FMOE_FUSED_GU_WARPS;          // dequantised gate/up GEMV warps
constexpr int kDownWarps = 16 - kGuWarps;              // down projection + combine warps
constexpr int kConsumerWarps = kGuWarps + kDownWarps;  // warps that hold the layer input
constexpr int kProducerWarp = kConsumerWarps;          // issues the bulk copies
constexpr int kFinalWarp = kConsumerWarps + 1;         // turns partial sums into h rows
constexpr int kExchangeWarp = kConsumerWarps + 2;      // gathers the h of even slots
constexpr int kExchangeWarp2 = kConsumerWarps + 3;     // routes; gathers the h of odd slots
constexpr int kRouteXw = 1;                            // the exchange warp (0, 1) that routes
constexpr int kFusedThreads = 32 * (kConsumerWarps + 4);
// registers per thread: the most that every warp can hold when the warps are
// spread over the SM's four schedulers, each with 16K registers (8 at a time)
constexpr int kFusedWarpsPerScheduler = (kFusedThreads / 32 + 3) / 4;
constexpr int kFusedMaxRegs = (16384 / (kFusedWarpsPerScheduler * 32)) / 8 * 8;
constexpr int kMaxFusedLayers = 64;    // layers per launch; longer stacks use several launches
constexpr int kMaxSlots = FMOE_MAX_TOPK + 1;
constexpr int kMaxStages = 16;
// Tuning of the persistent kernel (compile-time; the defaults are the
// measured best): ring stages at most, slots by which a slot's down records
// trail its gate/up records, whether an exchange warp waits for its own
// block's share of a slot before polling the other blocks' shares, whether
// the producer waits for the previous layer's last exchange before it
// requests the next layer's rows (its copies would otherwise queue ahead of
// the exchange's loads), and how the block's rows are split into bulk copies.
#ifndef FMOE_FUSED_STAGE_CAP
#define FMOE_FUSED_STAGE_CAP 16
#endif
#ifndef FMOE_FUSED_DOWN_LAG
#define FMOE_FUSED_DOWN_LAG 3
#endif
#ifndef FMOE_XCHG_WAIT_OWN
#define FMOE_XCHG_WAIT_OWN 1
#endif
#ifndef FMOE_FUSED_LATE_PREFETCH
#define FMOE_FUSED_LATE_PREFETCH 1
#endif
// Pause between two polls of published (value, tag) words: every block
// polls the same few lines of L2, so polling too often slows down the
// stores it is waiting for.
#ifndef FMOE_INPUT_POLL_NS
#define FMOE_INPUT_POLL_NS 32
#endif
#ifndef FMOE_EXCHANGE_POLL_NS
#define FMOE_EXCHANGE_POLL_NS 32
#endif
constexpr unsigned kInputPollNs = FMOE_INPUT_POLL_NS;
constexpr unsigned kExchangePollNs = FMOE_EXCHANGE_POLL_NS;
#ifndef FMOE_FUSED_TAIL_SLOTS
#define FMOE_FUSED_TAIL_SLOTS 2
#endif
constexpr int kFusedTailSlots = FMOE_FUSED_TAIL_SLOTS;   // last slots whose down rows the gate/up warps do
#ifndef FMOE_FUSED_ISSUE_LANES
#define FMOE_FUSED_ISSUE_LANES 4
#endif
constexpr int kFusedIssueLanes = FMOE_FUSED_ISSUE_LANES;   // producer lanes that take turns issuing copies
#ifndef FMOE_FUSED_ROWS_PER_COPY
#define FMOE_FUSED_ROWS_PER_COPY 64
#endif
#ifndef FMOE_FUSED_DOWN_COPIES
#define FMOE_FUSED_DOWN_COPIES 1
#endif
constexpr int kFusedRowsPerCopy = FMOE_FUSED_ROWS_PER_COPY;   // gate/up records per bulk copy
constexpr int kFusedDownCopies = FMOE_FUSED_DOWN_COPIES;      // bulk copies per slot's down records
constexpr int kFusedStageCap = FMOE_FUSED_STAGE_CAP < kMaxStages ? FMOE_FUSED_STAGE_CAP : kMaxStages;
constexpr int kFusedDownLag = FMOE_FUSED_DOWN_LAG;
constexpr int kMaxDownGroups = 8;      // down row groups per down warp
constexpr int kCtrlBytes = 2048;       // barriers, routing result, reductions, tail sums
constexpr int kMaxTailRows = (kCtrlBytes - 1536) / 4;   // down rows per block the tail sums can hold
constexpr int kMaxTailGroups = 4;      // down row groups per gate/up warp in the tail

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
  int rows_per_stage;       // gate/up rows per ring stage (two per consumer warp and slice range)
  int nstage, stage_bytes;  // ring
  int dslot_bytes;          // one slot's down records
  int nrmax, nparts;        // gate/up rows per block and partial sums per row
  int part_off, xs_off, stage_off, hs_off, hs_slot_bytes, darea_off, ring_off;
  int dlag;                 // a slot's down records are copied, and used, dlag slots after its gate/up
};

struct FusedParams {
  int bits, H, I, E, K, S, L;
  int norm;                 // 1: input = RMSNorm(hin), residual = hin (stack); 0: given x / residual
  float eps;
  size_t blob;
  BlobLayout lay;
  const float* x;           // norm == 0: input [H]
  const float* residual;    // norm == 0: residual [H]
  float* out;               // norm == 0: output [H];  norm == 1: h (in for layer 0, out for the last)
  const float* logits;      // [L][E]
  float* hmid;              // [K+S][I] h of the last layer (plain fp32)
  unsigned long long* hll;  // [K+S][I] (value, tag) exchange of h
  unsigned long long* hbufll;  // [2][H] (value, tag) outputs of layers 0..L-2 (stacks)
  int32_t* ids_out;         // [L][K] or nullptr
  float* w_out;             // [L][K] or nullptr
  float* gate_out;          // [L] or nullptr
  uint32_t* exit_ctr;       // zero on entry and on exit
  uint32_t* epoch;          // incremented by the last block out
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

cudaError_t launch_wait_test(uint32_t* counter, uint32_t* err, int n_blocks, int expected,
                             unsigned long long timeout_ns, cudaStream_t st);

}  // namespace fmoe
