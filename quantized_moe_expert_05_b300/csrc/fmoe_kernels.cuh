// Kernel argument structs and launcher declarations shared by the .cu files.
#pragma once

#include "fmoe_internal.cuh"

namespace fmoe {

// Arguments of the general kernels (fmoe_generic.cu).
struct GenericArgs {
  int bits, H, I, E, K, S, T;
  size_t blob;
  BlobLayout lay;
  const uint8_t* experts;
  const uint8_t* shared;
  const int32_t* ids;       // [T][K]
  const float* weights;     // [T][K]
  const float* gate;        // [T]
  const float* x;           // [T][H]
  const float* residual;    // [T][H]
  float* out;               // [T][H]
  float* h;                 // [T][K+S][I]
  uint32_t* err;
};

cudaError_t launch_route(const float* logits, int T, int E, int K, int32_t* ids, float* weights,
                         const uint16_t* wsg, const float* x, int H, float* gate, cudaStream_t st);
cudaError_t launch_gateup_generic(const GenericArgs& a, cudaStream_t st);
cudaError_t launch_down_y(const GenericArgs& a, float* y, cudaStream_t st);
cudaError_t launch_down_combine(const GenericArgs& a, cudaStream_t st);

// ---------------------------------------------------------------------------
// single-launch persistent kernel (fmoe_fused.cu)
// ---------------------------------------------------------------------------
constexpr int kGuWarps = 12;                           // dequantised gate/up GEMV warps
constexpr int kDownWarps = 4;                          // down projection + combine warps
constexpr int kConsumerWarps = kGuWarps + kDownWarps;  // warps that hold the layer input
constexpr int kProducerWarp = kConsumerWarps;          // issues the bulk copies
constexpr int kFinalWarp = kConsumerWarps + 1;         // turns partial sums into h rows
constexpr int kExchangeWarp = kConsumerWarps + 2;      // routes; gathers the h of even slots
constexpr int kExchangeWarp2 = kConsumerWarps + 3;     // gathers the h of odd slots
constexpr int kFusedThreads = 32 * (kConsumerWarps + 4);
// registers per thread: the most that every warp can hold when the warps are
// spread over the SM's four schedulers, each with 16K registers (8 at a time)
constexpr int kFusedWarpsPerScheduler = (kFusedThreads / 32 + 3) / 4;
constexpr int kFusedMaxRegs = (16384 / (kFusedWarpsPerScheduler * 32)) / 8 * 8;
constexpr int kMaxFusedLayers = 64;    // layers per launch; longer stacks use several launches
constexpr int kMaxSlots = FMOE_MAX_TOPK + 1;
constexpr int kMaxStages = 16;
constexpr int kMaxDownGroups = 8;      // down row groups per down warp
constexpr int kCtrlBytes = 1536;       // barriers, routing result, reductions

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
cudaError_t launch_fused(FusedParams& p, const FusedPlan& plan, cudaStream_t st);

cudaError_t launch_wait_test(uint32_t* counter, uint32_t* err, int n_blocks, int expected,
                             unsigned long long timeout_ns, cudaStream_t st);

}  // namespace fmoe
