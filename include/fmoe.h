/*
 * fmoe.h -- C ABI of the batch-1 quantised MoE expert block for B300 (sm_103a).
 *
 * The operations follow the flash-moe write-ups (discuss.pytorch.kr post
 * "flash-moe: C/Metal engine running a 397B MoE on an M3 Max" and GeekNews
 * topic 27758 "Flash-MoE - running a 397B-parameter model on a laptop"):
 *   - "per-layer pipeline": router logits -> softmax + top-K -> expert forward
 *     -> combine + residual (+ norm) feeding the next layer;
 *   - "FMA-optimised dequant kernel": expert weights are 4-bit (or 2-bit)
 *     codes dequantised as code * scale + bias;
 *   - "hand-written Metal compute shaders": dequant matvec, fused SwiGLU,
 *     two-stage RMSNorm, and one fused "MoE combine + residual + sigmoid gate";
 *   - "Qwen3.5-397B-A17B model architecture": K routed experts out of E plus
 *     one always-on shared expert.
 *
 * Conventions (all entry points):
 *   - Every pointer argument is a DEVICE pointer unless its comment says
 *     "host".  The caller owns all memory; the library allocates nothing and
 *     keeps no state between calls except inside the caller's workspace.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Calls enqueue work and return without synchronising, except
 *     fmoe_last_device_error, which synchronises `stream`.
 *   - Host-side argument checks return FMOE_ERR_INVALID_ARG (null or
 *     misaligned pointer, inconsistent sizes) or FMOE_ERR_UNSUPPORTED (a
 *     shape or bit width this build does not implement) and enqueue nothing.
 *     A failed launch returns FMOE_ERR_CUDA.  Device-side waits that run out
 *     of time set an error word in the workspace and return; the host reads
 *     it with fmoe_last_device_error (FMOE_ERR_TIMEOUT).
 *   - fp32 activations are read and written as IEEE binary32.  Router logits
 *     must be finite (NaN/inf logits give unspecified ids).  Activations must
 *     stay below 2^40 in magnitude (the dot products pre-scale x by powers of
 *     two; larger values overflow to inf).  The single-launch kernel (T = 1)
 *     adds the partial outputs of its blocks in fixed point with 2^-28
 *     resolution: a block's share of an output element beyond 2^19 in
 *     magnitude is clamped and reported (FMOE_ERR_RANGE from
 *     fmoe_last_device_error).
 *
 * Packed expert blob (one per expert, contiguous, 256-byte aligned):
 *   gate/up records, r = 0..I-1, each padded to a multiple of 16 bytes:
 *     gate_q  [H*bits/32] uint32   codes of gate row r; code c at bits
 *                                  (c mod 32/bits)*bits of word c/(32/bits)
 *                                  (lowest bits first)
 *     up_q    [H*bits/32] uint32   codes of up row r
 *     gate_sb [H/64]      uint32   bits 0..15 scale (bf16), 16..31 bias (bf16)
 *     up_sb   [H/64]      uint32
 *   the down projection by column, i = 0..I-1, from the next 256-byte
 *   boundary, H*bits/8 bytes each:
 *     down_q  [H*bits/32] uint32   codes of column i; row j at bits
 *                                  (j mod 32/bits)*bits of word j/(32/bits)
 *   its scale/bias words by group of 64 columns, g = 0..I/64-1, from the
 *   next 256-byte boundary, H words each:
 *     down_sb [H]         uint32   word j: row j's scale and bias for
 *                                  columns 64g .. 64g+63
 *   The dequantised weight of row r, column c of a matrix is q * scale[r][c/64]
 *   + bias[r][c/64]; gate/up rows have H columns, the down projection has H
 *   rows and I columns.  A range of gate/up rows (with their scales), a range
 *   of down columns and a range of down groups are each one contiguous byte
 *   range.  Blob size: fmoe_expert_bytes() (a multiple of 256); the routed
 *   experts of a layer sit at stride fmoe_expert_bytes() from `experts`.
 */
#ifndef FMOE_H
#define FMOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FMOE_OK = 0,
  FMOE_ERR_INVALID_ARG = 1,
  FMOE_ERR_UNSUPPORTED = 2,
  FMOE_ERR_CUDA = 3,
  FMOE_ERR_TIMEOUT = 4,
  FMOE_ERR_RANGE = 5
} fmoe_status;

/* Largest sizes this build accepts. */
#define FMOE_MAX_TOKENS 16      /* T per call                                  */
#define FMOE_MAX_TOPK 16        /* K routed experts per token                  */
#define FMOE_MAX_EXPERTS 1024   /* E routed experts per layer                  */
#define FMOE_MAX_HIDDEN 8192    /* H                                           */
#define FMOE_MAX_INTER 4096     /* I                                           */
#define FMOE_MAX_LAYERS 1024    /* L of fmoe_stack_decode                      */

/*
 * One MoE layer: describes caller-owned device memory (no ownership passes).
 *   bits          4 or 2
 *   group         quantisation group; must be 64
 *   hidden, inter H and I; multiples of 64 (H also a multiple of 128, I a
 *                 multiple of 128 for the fused single-launch path)
 *   n_experts     E routed experts stored at `experts`
 *   has_shared    0 or 1
 *   experts       E blobs at stride fmoe_expert_bytes(); 256-byte aligned
 *   shared        the shared expert's blob (256-byte aligned) or NULL
 *   shared_gate_w bf16[H] gate vector w_sg (bit patterns), or NULL if no shared
 */
typedef struct fmoe_layer {
  int32_t bits;
  int32_t group;
  int32_t hidden;
  int32_t inter;
  int32_t n_experts;
  int32_t has_shared;
  const void* experts;
  const void* shared;
  const uint16_t* shared_gate_w;
} fmoe_layer;

/* Bytes of one packed expert blob (0 for an unsupported shape). */
size_t fmoe_expert_bytes(int bits, int hidden, int inter, int group);

/*
 * Bytes of workspace a call needs for `layer`, T tokens, K routed experts and
 * L stacked layers (L = 1 for the single-block calls).  The workspace holds
 * intermediate activations, routing results, the batch plan, the device
 * error word and, in its first 256 + 24*H bytes (rounded up to a multiple of
 * 256), state that the single-launch kernel keeps between calls: a layer
 * count and three fixed-point accumulators of H 64-bit words through which
 * its blocks add up their partial outputs.  The workspace must be 256-byte
 * aligned and zeroed once before its first use (fmoe_workspace_init);
 * afterwards the library keeps it consistent.  Calls that share a workspace
 * must not overlap in time.
 */
size_t fmoe_workspace_bytes(const fmoe_layer* layer /* host */, int T, int K, int L);

/* Zero a workspace of `bytes` bytes (async on `stream`). */
fmoe_status fmoe_workspace_init(void* ws, size_t bytes, void* stream);

/*
 * Route T tokens: the flash-moe "softmax + top-K" step ("per-layer pipeline").
 *   logits  fp32 [T][E]   router logits (finite)
 *   ids     int32 [T][K]  out: the K largest logits per token in descending
 *                         order; equal logits rank the lower expert id first
 *                         (-0 and +0 are equal)
 *   weights fp32 [T][K]   out: softmax over the K selected logits (sums to 1)
 * 1 <= T <= FMOE_MAX_TOKENS, 1 <= K <= min(E, FMOE_MAX_TOPK), E <= FMOE_MAX_EXPERTS.
 */
fmoe_status fmoe_route(const float* logits, int T, int E, int K,
                       int32_t* ids, float* weights, void* stream);

/*
 * Router projection (flash-moe "per-layer pipeline": the second command
 * buffer computes the routing logits on the GPU):
 *   logits[t][e] = sum_j W_r[e][j] * x[t][j]
 *   w_router  bf16 [E][H]   router matrix (bf16 bit patterns), 16-byte aligned
 *   x         fp32 [T][H]   16-byte aligned
 *   logits    fp32 [T][E]   out; must not overlap x or w_router
 * 1 <= T <= FMOE_MAX_TOKENS, H a multiple of 64 up to FMOE_MAX_HIDDEN,
 * 1 <= E <= FMOE_MAX_EXPERTS.  The sums are taken in fp32 in a fixed order
 * (deterministic).  FMOE_ERR_INVALID_ARG for bad sizes or pointers.
 */
fmoe_status fmoe_router_logits(const uint16_t* w_router, const float* x, int T, int hidden, int E,
                               float* logits, void* stream);

/*
 * Routing from the layer input: fmoe_router_logits, then fmoe_route on the
 * logits and, when shared_gate_w is not null, gate[t] = sigmoid(w_sg . x[t])
 * (two launches on `stream`).
 *   logits  fp32 [T][E]   out (kept: the routing decisions are taken on them)
 *   ids, weights          out, as fmoe_route
 *   shared_gate_w bf16 [H] (16-byte aligned) or NULL; gate fp32 [T] out (NULL
 *                 when shared_gate_w is)
 */
fmoe_status fmoe_route_from_x(const uint16_t* w_router, const float* x, int T, int hidden, int E, int K,
                              const uint16_t* shared_gate_w, float* logits, int32_t* ids, float* weights,
                              float* gate, void* stream);

/*
 * The MoE-adjacent steps of a layer (flash-moe "per-layer pipeline": CMD2
 * runs o_proj and the norm on the GPU before the routing).
 *
 * fmoe_dense_row_bytes: bytes of one row record of a dense quantised matrix:
 *   the row's codes (hidden*bits/8 bytes, lowest bits first within each
 *   32-bit word), then one (scale,bias) word per 64 columns (scale bf16 in
 *   bits 0..15, bias bf16 in bits 16..31), padded to a multiple of 16 bytes.
 *   0 for a bad shape.
 * fmoe_dense_gemv: y[t][r] = sum_j (q[r][j]*s + b) * x[t][j] (+ residual[t][r])
 *   for a dense matrix of N row records (the o_proj: N = H); bits 4 or 2.
 *   w 16-byte aligned, N row records; x fp32 [T][H]; residual fp32 [T][N] or
 *   NULL, may be y (in-place residual add); y fp32 [T][N] must not overlap
 *   x or w.  1 <= T <= FMOE_MAX_TOKENS, H a multiple of 64 up to
 *   FMOE_MAX_HIDDEN, N >= 1.  Deterministic (fixed summation order).
 * fmoe_rmsnorm: x[t] = h[t] / sqrt(mean(h[t]^2) + eps) * weight (weight fp32
 *   [H], or NULL for unit weight); x may be h.
 */
size_t fmoe_dense_row_bytes(int bits, int hidden);
fmoe_status fmoe_dense_gemv(const void* w, int bits, int N, int hidden, const float* x, int T,
                            const float* residual, float* y, void* stream);
fmoe_status fmoe_rmsnorm(const float* h, const float* weight, int T, int hidden, float eps, float* x,
                         void* stream);

/*
 * Expert forward for given ids (flash-moe CMD3 "expert forward", without the
 * combine): for token t and slot k < K, y[t][k] = Wd (silu(Wg x_t) * (Wu x_t))
 * of routed expert ids[t][k]; if layer->has_shared, slot K holds the shared
 * expert's output for x_t.
 *   ids  int32 [T][K]         expert ids in [0, E)
 *   x    fp32  [T][H]
 *   y    fp32  [T][K+S][H]    out, unweighted (S = has_shared)
 *   ws   workspace of fmoe_workspace_bytes(layer, T, K, 1) bytes
 * Each distinct expert among the T*K ids (and the shared expert) is read
 * once, whatever the number of tokens that use it.  An id outside [0, E) is
 * not read: its y row is zero and the workspace error word records it
 * (fmoe_last_device_error then returns FMOE_ERR_INVALID_ARG).
 */
fmoe_status fmoe_expert_ffn(const fmoe_layer* layer /* host */, const int32_t* ids,
                            int T, int K, const float* x, float* y,
                            void* ws, void* stream);

/*
 * One MoE block (flash-moe: routing, expert forward, and the fused "MoE
 * combine + residual + sigmoid gate"):
 *   out[t] = residual[t] + sum_k w[t][k] * y[t][k] + sigmoid(w_sg . x[t]) * y_shared[t]
 * with (ids, w) = fmoe_route(router_logits[t]) and y as in fmoe_expert_ffn
 * (the sigmoid term only if layer->has_shared).
 *   x, residual, out  fp32 [T][H];  router_logits fp32 [T][E]
 *   out may alias residual; it must not overlap x or router_logits.
 * T = 1 runs as one persistent launch when the shape fits it (H/32 a power
 * of two, H >= 128); otherwise (and for every T > 1) four launches: plan,
 * gate/up, down, combine, in which each distinct expert among the T*K picks
 * is read once (see fmoe_ws_batch_plan).  The routing result is left in the workspace (see
 * fmoe_ws_routing).
 */
fmoe_status fmoe_moe_block(const fmoe_layer* layer /* host */, const float* x,
                           const float* router_logits, const float* residual,
                           float* out, int T, int K, void* ws, void* stream);

/*
 * One decode token through L pre-norm MoE blocks (flash-moe "deferred CMD3":
 * combine, residual and normalisation stay on the GPU and feed the next
 * layer; the RMSNorm is the write-ups' two-stage RMS normalisation with unit
 * weight):
 *   for l in 0..L-1:  h <- h + MoE_l(h / sqrt(mean(h^2) + eps))
 * where MoE_l routes with logits[l] and uses residual 0 (the block's
 * residual is h itself).
 *   layers  host array of L layer descriptors, all with the same bits,
 *           hidden, inter, n_experts and has_shared
 *   logits  fp32 [L][E];  h fp32 [H] in/out
 *   ws      workspace of fmoe_workspace_bytes(&layers[0], 1, K, L) bytes
 * No layer's routed experts are read before the previous layer's output is
 * complete (their ids depend on it); a layer's shared expert, whose identity
 * is fixed, may be requested as soon as the reading block has finished its
 * share of the previous layer.  Shapes the single-launch kernel takes run as
 * one launch per 64 layers; other shapes run per layer as an RMSNorm launch
 * followed by the batched block.  The routing result of layer l is left at
 * row l of the workspace's ids/weights/gate (fmoe_ws_routing with T = L).
 */
fmoe_status fmoe_stack_decode(const fmoe_layer* layers /* host */, int L,
                              const float* logits, float* h, int K, float eps,
                              void* ws, void* stream);

/*
 * Device pointers, inside a workspace, to the routing result of the last
 * fmoe_moe_block call (ids int32 [T][K], weights fp32 [T][K], gate fp32 [T]
 * = sigmoid(w_sg . x) or 0 without a shared expert) and to the
 * intermediate activations h fp32 [T][K+S][I].  Host function; no sync.
 */
fmoe_status fmoe_ws_routing(void* ws, const fmoe_layer* layer /* host */, int T, int K,
                            int32_t** ids, float** weights, float** gate, float** h);

/*
 * Device pointer, inside a workspace, to the batch plan written by the last
 * fmoe_expert_ffn call or batched fmoe_moe_block call (T > 1) on it:
 *   plan[0]  number of items;  plan[1]  distinct experts read (shared incl.)
 *   item i at plan + 8 + 8*i:  [0] expert id (-1: shared expert)
 *                              [1] n, the item's tokens (1..4)
 *                              [2+g], g < n: (t << 8) | slot of token g
 * A distinct expert picked by m tokens has ceil(m/G) items (G = 4, or 2 or 1
 * for shapes whose staged inputs leave no room for four tokens), listed in
 * order of first appearance in ids (token-major); its codes are read from
 * HBM once.
 * Diagnostic; host function, no sync.
 */
fmoe_status fmoe_ws_batch_plan(void* ws, const fmoe_layer* layer /* host */, int T, int K, int32_t** plan);

/*
 * Test hook (host arithmetic only; no CUDA call): the launch geometry the
 * library would use for a layer shape on a device with `sms` SMs and
 * `smem_max` bytes of opt-in shared memory per block.  Writes FMOE_GEO_COUNT
 * int64 values to `out` (indices below; byte counts and offsets of the
 * persistent kernel's and the batched kernels' shared memory).  Returns
 * FMOE_ERR_INVALID_ARG if out is null or n < FMOE_GEO_COUNT.
 */
enum {
  FMOE_GEO_FUSED_OK, FMOE_GEO_FUSED_GRID, FMOE_GEO_FUSED_SMEM, FMOE_GEO_FUSED_CTRL_BYTES,
  FMOE_GEO_FUSED_XS_OFF, FMOE_GEO_FUSED_PART_OFF, FMOE_GEO_FUSED_HBUF_OFF, FMOE_GEO_FUSED_HBUF_STRIDE,
  FMOE_GEO_FUSED_DSCR_OFF, FMOE_GEO_FUSED_DAREA_OFF, FMOE_GEO_FUSED_DAREA_BYTES, FMOE_GEO_FUSED_RING_OFF,
  FMOE_GEO_FUSED_NSTAGE,
  FMOE_GEO_FUSED_STAGE_BYTES, FMOE_GEO_FUSED_ROWS_PER_STAGE, FMOE_GEO_FUSED_NPARTS, FMOE_GEO_FUSED_LEN_MAX,
  FMOE_GEO_BATCH_GRID, FMOE_GEO_BATCH_G, FMOE_GEO_BATCH_GU_WARPS, FMOE_GEO_BATCH_GU_ROWS,
  FMOE_GEO_BATCH_GU_NSTAGE, FMOE_GEO_BATCH_GU_STAGE_BYTES, FMOE_GEO_BATCH_GU_XS_BYTES, FMOE_GEO_BATCH_GU_SMEM,
  FMOE_GEO_BATCH_D_ROWS, FMOE_GEO_BATCH_D_H_BYTES, FMOE_GEO_BATCH_D_SMEM, FMOE_GEO_BATCH_CTRL_BYTES,
  FMOE_GEO_COUNT
};
fmoe_status fmoe_debug_launch_geometry(int bits, int hidden, int inter, int K, int has_shared, int sms,
                                       int smem_max, int64_t* out, int n);

/*
 * Test hook (host arithmetic only; no CUDA call): the intermediate columns
 * that block `block` of `sms` owns in the single-launch kernel, as pieces of
 * one slot each.  Writes out[0] = the number of pieces and, for piece q,
 * out[1+8q .. 8+8q] = slot (0 = the shared expert when has_shared), first
 * column, column count, first local index, byte offsets of its codes and of
 * its (scale,bias) words in the block's down area, first 64-column group,
 * group count.  n must be at least 33.  FMOE_ERR_INVALID_ARG for a bad shape
 * or block.
 */
fmoe_status fmoe_debug_block_pieces(int bits, int hidden, int inter, int K, int has_shared, int sms,
                                    int block, int64_t* out, int n);

/*
 * Expert slot pool: n_slots HBM slots of one expert blob each, filled from a
 * copy of all n_experts blobs in pinned host memory (host memory stands in
 * for the SSD of the flash-moe write-up, section "SSD expert streaming and
 * 'Trust the OS'"; fixed slots with eviction as in the slotstream write-up,
 * "10 of 512 experts per layer"; whole-expert copies, "the disk was not the
 * slow part").  All calls but fmoe_pool_load are host code that touch no
 * device.  A routing step goes:
 *   1. ids of the step's T*K picks on the host (e.g. fmoe_route, then a copy);
 *   2. fmoe_pool_plan(ids) -> the slot of each pick and the loads (misses);
 *   3. fmoe_pool_load(loads, copy_stream): one cudaMemcpyAsync per miss;
 *   4. fmoe_pool_slot_logits -> logits over slots (the picks keep their
 *      logits, every other slot gets -FLT_MAX);
 *   5. fmoe_moe_block with layer.experts = the slots, layer.n_experts =
 *      n_slots and the slot logits, on a stream ordered after step 3.
 * Top-K and softmax over the slot logits select exactly the planned slots
 * with the same weights.
 *
 * fmoe_pool_state_bytes: host bytes of the pool's bookkeeping (0 for bad
 *   sizes).  The caller owns that memory (8-byte aligned), the device slots
 *   (n_slots * blob_bytes, 256-byte aligned) and the pinned host blobs
 *   (n_experts * blob_bytes, expert e at e * blob_bytes).
 * fmoe_pool_init: empty pool; FMOE_ERR_INVALID_ARG for bad sizes/pointers.
 * fmoe_pool_plan: for the n expert ids of one request (duplicates allowed),
 *   the slot of each in slots[n]; each distinct expert not resident gets the
 *   least recently used slot that neither this request nor the `keep`
 *   requests before it used (an empty slot first, ties to the lower slot),
 *   listed as (expert, slot) in loads[2*n_loads].  Slots of a request whose
 *   compute may still be running must be kept (keep >= 1) or their loads
 *   ordered after that compute.  FMOE_ERR_INVALID_ARG (nothing changed) for
 *   an id outside [0, n_experts) or a request needing more slots than are
 *   free to evict.
 * fmoe_pool_load: the copies of `loads` on `stream`.
 * fmoe_pool_slot_logits: slot_logits [T][n_slots] from logits [T][n_experts]
 *   and the request's ids / slots [T][K] (all host).
 * fmoe_pool_stats: distinct experts found resident (hits) and loaded
 *   (misses) over all requests, and the number of requests.
 * The write-ups' own reads go to SSD and the OS page cache; this pool is the
 * HBM counterpart, not a port of either.
 */
size_t fmoe_pool_state_bytes(int n_slots, int n_experts);
fmoe_status fmoe_pool_init(void* state /* host */, size_t state_bytes, int n_slots, int n_experts,
                           size_t blob_bytes, void* slots_dev, const void* host_blobs);
fmoe_status fmoe_pool_plan(void* state, const int32_t* ids /* host */, int n, int keep,
                           int32_t* slots /* host */, int32_t* loads /* host [2n] */, int* n_loads);
fmoe_status fmoe_pool_load(void* state, const int32_t* loads /* host */, int n_loads, void* stream);
fmoe_status fmoe_pool_slot_logits(const void* state, const float* logits /* host */,
                                  const int32_t* ids /* host */, const int32_t* slots /* host */, int T, int K,
                                  float* slot_logits /* host */);
fmoe_status fmoe_pool_stats(const void* state, uint64_t* hits, uint64_t* misses, uint64_t* requests);

/* Static description of a status code (host). */
const char* fmoe_status_string(fmoe_status s);

/*
 * Synchronise `stream`, then read and clear the workspace's device error
 * word: FMOE_OK; FMOE_ERR_TIMEOUT if a device-side wait gave up since the
 * last call; FMOE_ERR_INVALID_ARG if fmoe_expert_ffn met an expert id
 * outside [0, E); FMOE_ERR_RANGE if a partial sum left the fixed-point
 * range.  After a timeout the workspace must be re-initialised with
 * fmoe_workspace_init before reuse.
 */
fmoe_status fmoe_last_device_error(void* ws, void* stream);

/*
 * Test hook for the bounded device-side waits: launches `n_blocks` blocks
 * that arrive at a workspace counter and wait for `expected` arrivals for at
 * most `timeout_us` microseconds.  With expected > n_blocks the wait runs
 * out and the error word is set (no trap, no hang); with expected ==
 * n_blocks it completes.  1 <= n_blocks <= 148 * 4.
 */
fmoe_status fmoe_debug_wait_test(void* ws, int n_blocks, int expected,
                                 int timeout_us, void* stream);

/*
 * Bytes of the library's own scratch array used by fmoe_moe_block_noalloc.
 * Every GPU that loads the library holds this much device memory for it
 * until the process exits.
 */
#define FMOE_NOALLOC_SCRATCH_BYTES (128u * 1024u)

/*
 * fmoe_moe_block for one token (T = 1) without a caller workspace.
 *
 * The flash-moe write-ups have no counterpart to this call; it exists for
 * callers that cannot allocate device memory (code running inside an
 * allocator or memory-pool callback, plugins whose host framework owns all
 * device allocations, real-time loops that must not block in cudaMalloc).
 * Instead of a workspace it uses a fixed array of FMOE_NOALLOC_SCRATCH_BYTES
 * bytes that the library declares in device memory.  It calls no cudaMalloc,
 * cudaFree or other allocating routine.
 *
 *   layer, x, router_logits, residual, out, K
 *                 as fmoe_moe_block with T = 1 (out may alias residual)
 *   device_error  device pointer to one uint32, or NULL: after the block, the
 *                 call copies the kernel's error word there (0 = no error;
 *                 nonzero = a device-side wait timed out and `out` is not
 *                 valid).  Written asynchronously on `stream`.
 *
 * Returns FMOE_ERR_INVALID_ARG (and enqueues nothing) for the argument
 * errors of fmoe_moe_block and when the kernel's scratch (256 + 24*H bytes,
 * rounded up to 256: 98,560 bytes at H = 4096, so H up to 5,440) exceeds
 * FMOE_NOALLOC_SCRATCH_BYTES; FMOE_ERR_UNSUPPORTED for shapes the
 * single-launch kernel does not cover; FMOE_ERR_CUDA if the set-up or a
 * launch fails.
 *
 * Each call asks the runtime for the array's device address on the current
 * device (cudaGetSymbolAddress); the first call on a device loads the
 * library's device code there, so make that first call before any stream
 * capture.  Every call on a device uses the same array and clears it (its
 * error word, counters and accumulators) before its launch: calls that
 * overlap on the GPU (other streams, or other host threads) race on it and
 * must be serialised by the caller.  The routing result is not kept.
 */
fmoe_status fmoe_moe_block_noalloc(const fmoe_layer* layer /* host */, const float* x,
                                   const float* router_logits, const float* residual,
                                   float* out, int K, uint32_t* device_error,
                                   void* stream);

#ifdef __cplusplus
}
#endif
#endif /* FMOE_H */
