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
constexpr int kFusedThreads = 512;
constexpr int kMaxFusedLayers = 64;    // layers per launch; longer stacks use several launches
constexpr int kMaxSlots = FMOE_MAX_TOPK + 1;
constexpr int kMaxStages = 16;
constexpr int kMaxRowsPerTeam = 4;     // down rows per team per block

struct FusedLayerPtrs {
  const uint8_t* experts;
  const uint8_t* shared;
  const uint16_t* wsg;
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
  float* hmid;              // [K+S][I]
  float* hbuf;              // [2][H]
  int32_t* ids_out;         // [L][K] or nullptr
  float* w_out;             // [L][K] or nullptr
  float* gate_out;          // [L] or nullptr
  uint32_t* counters;       // [L][K+S+1] + 1 exit counter (zero on entry, zero on exit)
  uint32_t* err;
  unsigned long long timeout_ns;
  int copy_back;            // norm == 1 and L == 1: the result goes through hbuf then to out
  // shared-memory plan (host computed)
  int nstage, stage_bytes, dslot_bytes;
  int gu_cap_q, gu_cap_sb, d_cap_q, d_cap_sb;
  FusedLayerPtrs layer[kMaxFusedLayers];
};

struct FusedPlan {
  bool ok;
  int grid;
  size_t smem;
  int nstage, stage_bytes, dslot_bytes;
  int gu_cap_q, gu_cap_sb, d_cap_q, d_cap_sb;
};

// Plan the persistent launch for a shape; ok == false if the shape does not
// fit the kernel's limits (the caller then uses the general kernels).
FusedPlan fused_plan(int bits, int H, int I, int K, int S, int device);
cudaError_t launch_fused(FusedParams& p, const FusedPlan& plan, cudaStream_t st);

cudaError_t launch_wait_test(uint32_t* counter, uint32_t* err, int n_blocks, int expected,
                             unsigned long long timeout_ns, cudaStream_t st);

}  // namespace fmoe
