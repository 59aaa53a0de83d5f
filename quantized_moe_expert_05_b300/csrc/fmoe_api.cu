// extern "C" entry points of libfmoe: argument checks, workspace carving and
// dispatch to the kernels.  See include/fmoe.h for the contract of each call.
#include <cstdio>
#include <cstring>

#include "fmoe_kernels.cuh"

using namespace fmoe;

namespace {

constexpr unsigned long long kTimeoutNs = 200ull * 1000 * 1000;   // 200 ms per device-side wait

bool aligned(const void* p, size_t a) { return host_aligned(p, a); }

fmoe_status from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return FMOE_OK;
  cudaGetLastError();   // clear a sticky launch error so later calls start clean
  return FMOE_ERR_CUDA;
}

struct Ws {
  WsLayout lay;
  uint8_t* base;
  uint32_t* err() const { return reinterpret_cast<uint32_t*>(base + lay.err); }
  uint32_t* exit_ctr() const { return reinterpret_cast<uint32_t*>(base + lay.exit_ctr); }
  uint32_t* lbase() const { return reinterpret_cast<uint32_t*>(base + lay.lbase); }
  unsigned long long* acc() const { return reinterpret_cast<unsigned long long*>(base + lay.acc); }
  int32_t* ids() const { return reinterpret_cast<int32_t*>(base + lay.ids); }
  float* weights() const { return reinterpret_cast<float*>(base + lay.weights); }
  float* gate() const { return reinterpret_cast<float*>(base + lay.gate); }
  float* h() const { return reinterpret_cast<float*>(base + lay.h); }
  float* y() const { return reinterpret_cast<float*>(base + lay.y); }
  float* xn() const { return reinterpret_cast<float*>(base + lay.xn); }
  int32_t* plan() const { return reinterpret_cast<int32_t*>(base + lay.plan); }
};

Ws carve(void* ws, const fmoe_layer* L, int T, int K, int n_layers) {
  Ws w;
  w.lay = ws_layout(L->hidden, L->inter, L->has_shared, T > n_layers ? T : n_layers, K, n_layers);
  w.base = static_cast<uint8_t*>(ws);
  return w;
}

BatchArgs batch_args(const fmoe_layer* L, int T, int K, const Ws& w) {
  BatchArgs a{};
  a.bits = L->bits;
  a.H = L->hidden;
  a.I = L->inter;
  a.E = L->n_experts;
  a.K = K;
  a.S = L->has_shared;
  a.T = T;
  a.lay = blob_layout(L->bits, L->hidden, L->inter);
  a.blob = a.lay.bytes;
  a.experts = static_cast<const uint8_t*>(L->experts);
  a.shared = static_cast<const uint8_t*>(L->shared);
  a.ids = w.ids();
  a.weights = w.weights();
  a.gate = w.gate();
  a.h = w.h();
  a.y = w.y();
  a.plan = w.plan();
  a.err = w.err();
  a.timeout_ns = kTimeoutNs;
  return a;
}

// The workspace fields of the persistent kernel.
void fused_ws(FusedParams& p, const Ws& w) {
  p.hmid = w.h();
  p.acc = w.acc();
  p.lbase = w.lbase();
  p.exit_ctr = w.exit_ctr();
  p.err = w.err();
  p.timeout_ns = kTimeoutNs;
}

int current_device() {
  int d = 0;
  cudaGetDevice(&d);
  return d;
}

}  // namespace

extern "C" {

size_t fmoe_expert_bytes(int bits, int hidden, int inter, int group) {
  if ((bits != 4 && bits != 2) || group != kGroup) return 0;
  if (hidden <= 0 || inter <= 0 || hidden % kGroup || inter % kGroup) return 0;
  return blob_layout(bits, hidden, inter).bytes;
}

size_t fmoe_workspace_bytes(const fmoe_layer* layer, int T, int K, int L) {
  if (layer == nullptr || T < 1 || K < 1 || L < 1) return 0;
  if (check_layer(layer, false) != FMOE_OK) return 0;
  return ws_layout(layer->hidden, layer->inter, layer->has_shared, T > L ? T : L, K, L).bytes;
}

fmoe_status fmoe_workspace_init(void* ws, size_t bytes, void* stream) {
  if (ws == nullptr || !aligned(ws, 256) || bytes == 0) return FMOE_ERR_INVALID_ARG;
  return from_cuda(cudaMemsetAsync(ws, 0, bytes, static_cast<cudaStream_t>(stream)));
}

fmoe_status fmoe_route(const float* logits, int T, int E, int K, int32_t* ids, float* weights, void* stream) {
  if (!host_vec_ok(logits) || ids == nullptr || weights == nullptr) return FMOE_ERR_INVALID_ARG;
  if (!aligned(ids, 4) || !aligned(weights, 4)) return FMOE_ERR_INVALID_ARG;
  if (T < 1 || T > FMOE_MAX_TOKENS || E < 1 || E > FMOE_MAX_EXPERTS) return FMOE_ERR_INVALID_ARG;
  if (K < 1 || K > E || K > FMOE_MAX_TOPK) return FMOE_ERR_INVALID_ARG;
  return from_cuda(launch_route(logits, T, E, K, ids, weights, nullptr, nullptr, 0, nullptr,
                                static_cast<cudaStream_t>(stream)));
}

fmoe_status fmoe_router_logits(const uint16_t* w_router, const float* x, int T, int hidden, int E, float* logits,
                               void* stream) {
  if (!host_vec_ok(w_router) || !host_vec_ok(x) || logits == nullptr || !aligned(logits, 4))
    return FMOE_ERR_INVALID_ARG;
  if (T < 1 || T > FMOE_MAX_TOKENS || E < 1 || E > FMOE_MAX_EXPERTS) return FMOE_ERR_INVALID_ARG;
  if (hidden <= 0 || hidden % kGroup || hidden > FMOE_MAX_HIDDEN) return FMOE_ERR_INVALID_ARG;
  const size_t lb = (size_t)T * E * 4;
  if (host_overlap(logits, lb, x, (size_t)T * hidden * 4) || host_overlap(logits, lb, w_router, (size_t)E * hidden * 2))
    return FMOE_ERR_INVALID_ARG;
  return from_cuda(launch_router(w_router, x, T, hidden, E, logits, static_cast<cudaStream_t>(stream)));
}

fmoe_status fmoe_route_from_x(const uint16_t* w_router, const float* x, int T, int hidden, int E, int K,
                              const uint16_t* shared_gate_w, float* logits, int32_t* ids, float* weights, float* gate,
                              void* stream) {
  if (ids == nullptr || weights == nullptr || !aligned(ids, 4) || !aligned(weights, 4)) return FMOE_ERR_INVALID_ARG;
  if (K < 1 || K > E || K > FMOE_MAX_TOPK) return FMOE_ERR_INVALID_ARG;
  if ((shared_gate_w == nullptr) != (gate == nullptr)) return FMOE_ERR_INVALID_ARG;
  if (shared_gate_w != nullptr && (!aligned(shared_gate_w, 16) || !aligned(gate, 4))) return FMOE_ERR_INVALID_ARG;
  fmoe_status s = fmoe_router_logits(w_router, x, T, hidden, E, logits, stream);
  if (s != FMOE_OK) return s;
  return from_cuda(launch_route(logits, T, E, K, ids, weights, shared_gate_w, x, hidden, gate,
                                static_cast<cudaStream_t>(stream)));
}

size_t fmoe_dense_row_bytes(int bits, int hidden) {
  if ((bits != 4 && bits != 2) || hidden <= 0 || hidden % kGroup || hidden > FMOE_MAX_HIDDEN) return 0;
  return (size_t)dense_row_bytes(bits, hidden);
}

fmoe_status fmoe_dense_gemv(const void* w, int bits, int N, int hidden, const float* x, int T, const float* residual,
                            float* y, void* stream) {
  if (fmoe_dense_row_bytes(bits, hidden) == 0 || N < 1 || T < 1 || T > FMOE_MAX_TOKENS) return FMOE_ERR_INVALID_ARG;
  if (!host_vec_ok(w) || !host_vec_ok(x) || y == nullptr || !aligned(y, 4)) return FMOE_ERR_INVALID_ARG;
  if (residual != nullptr && !aligned(residual, 4)) return FMOE_ERR_INVALID_ARG;
  const size_t yb = (size_t)T * N * 4;
  if (host_overlap(y, yb, x, (size_t)T * hidden * 4) ||
      host_overlap(y, yb, w, (size_t)N * dense_row_bytes(bits, hidden)))
    return FMOE_ERR_INVALID_ARG;
  if (residual != nullptr && residual != y && host_overlap(y, yb, residual, yb)) return FMOE_ERR_INVALID_ARG;
  return from_cuda(launch_dense_gemv(static_cast<const uint8_t*>(w), bits, N, hidden, x, T, residual, y,
                                     static_cast<cudaStream_t>(stream)));
}

fmoe_status fmoe_rmsnorm(const float* h, const float* weight, int T, int hidden, float eps, float* x, void* stream) {
  if (h == nullptr || x == nullptr || !aligned(h, 4) || !aligned(x, 4)) return FMOE_ERR_INVALID_ARG;
  if (weight != nullptr && !aligned(weight, 4)) return FMOE_ERR_INVALID_ARG;
  if (T < 1 || T > FMOE_MAX_TOKENS || hidden < 1 || hidden > FMOE_MAX_HIDDEN || !(eps >= 0.f))
    return FMOE_ERR_INVALID_ARG;
  const size_t hb = (size_t)T * hidden * 4;
  if (x != h && host_overlap(x, hb, h, hb)) return FMOE_ERR_INVALID_ARG;
  return from_cuda(launch_rmsnorm_w(h, weight, T, hidden, eps, x, static_cast<cudaStream_t>(stream)));
}

fmoe_status fmoe_expert_ffn(const fmoe_layer* layer, const int32_t* ids, int T, int K, const float* x, float* y,
                            void* ws, void* stream) {
  fmoe_status s = check_layer(layer, true);
  if (s != FMOE_OK) return s;
  if (T < 1 || T > FMOE_MAX_TOKENS || K < 1 || K > FMOE_MAX_TOPK || K > layer->n_experts)
    return FMOE_ERR_INVALID_ARG;
  if (ids == nullptr || !aligned(ids, 4) || !host_vec_ok(x) || !host_vec_ok(y) || ws == nullptr || !aligned(ws, 256))
    return FMOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  Ws w = carve(ws, layer, T, K, 1);
  BatchArgs a = batch_args(layer, T, K, w);
  a.ids_in = ids;
  a.x = x;
  a.y = y;
  return from_cuda(launch_batch(a, y, st));
}

fmoe_status fmoe_moe_block(const fmoe_layer* layer, const float* x, const float* router_logits,
                           const float* residual, float* out, int T, int K, void* ws, void* stream) {
  fmoe_status s = check_layer(layer, true);
  if (s != FMOE_OK) return s;
  if (T < 1 || T > FMOE_MAX_TOKENS || K < 1 || K > FMOE_MAX_TOPK || K > layer->n_experts)
    return FMOE_ERR_INVALID_ARG;
  if (ws == nullptr || !aligned(ws, 256)) return FMOE_ERR_INVALID_ARG;
  s = check_block_args(layer, x, router_logits, residual, out, T);
  if (s != FMOE_OK) return s;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  Ws w = carve(ws, layer, T, K, 1);
  const int S = layer->has_shared;

  if (T == 1) {
    FusedPlan pl = fused_plan(layer->bits, layer->hidden, layer->inter, K, S, current_device());
    if (pl.ok) {
      FusedParams p{};
      fused_params_for(p, layer, 1, K);
      fused_ws(p, w);
      p.norm = 0;
      p.eps = 0.f;
      p.x = x;
      p.residual = residual;
      p.out = out;
      p.logits = router_logits;
      p.ids_out = w.ids();
      p.w_out = w.weights();
      p.gate_out = w.gate();
      return from_cuda(launch_fused(p, pl, st));
    }
  }
  // batched path: plan (route, shared gate, distinct experts), gate/up +
  // SwiGLU, down, combine
  BatchArgs a = batch_args(layer, T, K, w);
  a.logits = router_logits;
  a.wsg = S ? layer->shared_gate_w : nullptr;
  a.x = x;
  a.residual = residual;
  a.out = out;
  return from_cuda(launch_batch(a, a.y, st));
}

fmoe_status fmoe_stack_decode(const fmoe_layer* layers, int L, const float* logits, float* h, int K, float eps,
                              void* ws, void* stream) {
  if (layers == nullptr || L < 1 || L > FMOE_MAX_LAYERS) return FMOE_ERR_INVALID_ARG;
  fmoe_status s = check_layer(&layers[0], true);
  if (s != FMOE_OK) return s;
  for (int l = 1; l < L; ++l) {
    s = check_layer(&layers[l], true);
    if (s != FMOE_OK) return s;
    if (layers[l].bits != layers[0].bits || layers[l].hidden != layers[0].hidden ||
        layers[l].inter != layers[0].inter || layers[l].n_experts != layers[0].n_experts ||
        layers[l].has_shared != layers[0].has_shared)
      return FMOE_ERR_INVALID_ARG;
  }
  if (K < 1 || K > FMOE_MAX_TOPK || K > layers[0].n_experts) return FMOE_ERR_INVALID_ARG;
  if (!host_vec_ok(logits) || !host_vec_ok(h) || ws == nullptr || !aligned(ws, 256)) return FMOE_ERR_INVALID_ARG;
  if (!(eps >= 0.f)) return FMOE_ERR_INVALID_ARG;
  const fmoe_layer& L0 = layers[0];
  const int S = L0.has_shared;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  Ws w = carve(ws, &L0, 1, K, L);
  FusedPlan pl = fused_plan(L0.bits, L0.hidden, L0.inter, K, S, current_device());
  if (pl.ok) {
    for (int l0 = 0; l0 < L; l0 += kMaxFusedLayers) {
      const int n = (L - l0) < kMaxFusedLayers ? (L - l0) : kMaxFusedLayers;
      FusedParams p{};
      fused_params_for(p, layers + l0, n, K);
      fused_ws(p, w);
      p.norm = 1;
      p.eps = eps;
      p.x = nullptr;
      p.residual = nullptr;
      p.out = h;
      p.logits = logits + (size_t)l0 * L0.n_experts;
      p.ids_out = w.ids() + (size_t)l0 * K;
      p.w_out = w.weights() + (size_t)l0 * K;
      p.gate_out = w.gate() + l0;
      cudaError_t e = launch_fused(p, pl, st);
      if (e != cudaSuccess) return from_cuda(e);
    }
    return FMOE_OK;
  }
  // general path (shapes the persistent kernel does not take): per layer an
  // RMSNorm launch, then the batched block with residual and output h
  for (int l = 0; l < L; ++l) {
    cudaError_t e = launch_rmsnorm(h, w.xn(), L0.hidden, eps, st);
    if (e != cudaSuccess) return from_cuda(e);
    BatchArgs a = batch_args(&layers[l], 1, K, w);
    a.logits = logits + (size_t)l * L0.n_experts;
    a.wsg = S ? layers[l].shared_gate_w : nullptr;
    a.ids = w.ids() + (size_t)l * K;
    a.weights = w.weights() + (size_t)l * K;
    a.gate = w.gate() + l;
    a.x = w.xn();
    a.residual = h;
    a.out = h;
    e = launch_batch(a, a.y, st);
    if (e != cudaSuccess) return from_cuda(e);
  }
  return FMOE_OK;
}

fmoe_status fmoe_ws_routing(void* ws, const fmoe_layer* layer, int T, int K, int32_t** ids, float** weights,
                            float** gate, float** h) {
  if (ws == nullptr || layer == nullptr || T < 1 || K < 1) return FMOE_ERR_INVALID_ARG;
  if (check_layer(layer, false) != FMOE_OK) return FMOE_ERR_INVALID_ARG;
  Ws w = carve(ws, layer, T, K, 1);
  if (ids) *ids = w.ids();
  if (weights) *weights = w.weights();
  if (gate) *gate = w.gate();
  if (h) *h = w.h();
  return FMOE_OK;
}

fmoe_status fmoe_ws_batch_plan(void* ws, const fmoe_layer* layer, int T, int K, int32_t** plan) {
  if (ws == nullptr || layer == nullptr || plan == nullptr || T < 1 || K < 1) return FMOE_ERR_INVALID_ARG;
  if (check_layer(layer, false) != FMOE_OK) return FMOE_ERR_INVALID_ARG;
  *plan = carve(ws, layer, T, K, 1).plan();
  return FMOE_OK;
}

fmoe_status fmoe_debug_launch_geometry(int bits, int hidden, int inter, int K, int has_shared, int sms,
                                       int smem_max, int64_t* out, int n) {
  if (out == nullptr || n < FMOE_GEO_COUNT) return FMOE_ERR_INVALID_ARG;
  for (int i = 0; i < FMOE_GEO_COUNT; ++i) out[i] = 0;
  if ((bits != 4 && bits != 2) || hidden <= 0 || inter <= 0 || hidden % kGroup || inter % kGroup)
    return FMOE_OK;
  const FusedPlan f = fused_plan_for(bits, hidden, inter, K, has_shared, sms, smem_max);
  out[FMOE_GEO_FUSED_OK] = f.ok ? 1 : 0;
  out[FMOE_GEO_FUSED_GRID] = f.grid;
  out[FMOE_GEO_FUSED_SMEM] = (int64_t)f.smem;
  out[FMOE_GEO_FUSED_CTRL_BYTES] = kCtrlBytes;
  out[FMOE_GEO_FUSED_XS_OFF] = f.xs_off;
  out[FMOE_GEO_FUSED_PART_OFF] = f.part_off;
  out[FMOE_GEO_FUSED_HBUF_OFF] = f.hbuf_off;
  out[FMOE_GEO_FUSED_HBUF_STRIDE] = f.hb;
  out[FMOE_GEO_FUSED_DSCR_OFF] = f.dscr_off;
  out[FMOE_GEO_FUSED_DAREA_OFF] = f.darea_off;
  out[FMOE_GEO_FUSED_DAREA_BYTES] = f.darea_bytes;
  out[FMOE_GEO_FUSED_RING_OFF] = f.ring_off;
  out[FMOE_GEO_FUSED_NSTAGE] = f.nstage;
  out[FMOE_GEO_FUSED_STAGE_BYTES] = f.stage_bytes;
  out[FMOE_GEO_FUSED_ROWS_PER_STAGE] = f.R;
  out[FMOE_GEO_FUSED_NPARTS] = f.nparts;
  out[FMOE_GEO_FUSED_LEN_MAX] = f.len_max;
  const BatchGeom g = batch_geometry_for(bits, hidden, inter, sms, smem_max);
  out[FMOE_GEO_BATCH_GRID] = g.grid;
  out[FMOE_GEO_BATCH_G] = g.G;
  out[FMOE_GEO_BATCH_GU_WARPS] = g.gu_warps;
  out[FMOE_GEO_BATCH_GU_ROWS] = g.gu_rows;
  out[FMOE_GEO_BATCH_GU_NSTAGE] = g.gu_nstage;
  out[FMOE_GEO_BATCH_GU_STAGE_BYTES] = g.gu_stage_bytes;
  out[FMOE_GEO_BATCH_GU_XS_BYTES] = g.gu_xs_bytes;
  out[FMOE_GEO_BATCH_GU_SMEM] = (int64_t)g.gu_smem;
  out[FMOE_GEO_BATCH_D_ROWS] = 32 * (32 / bits);
  out[FMOE_GEO_BATCH_D_H_BYTES] = g.bd_h_bytes;
  out[FMOE_GEO_BATCH_D_SMEM] = (int64_t)g.bd_smem;
  out[FMOE_GEO_BATCH_CTRL_BYTES] = kBatchCtrlBytes;
  return FMOE_OK;
}

fmoe_status fmoe_debug_block_pieces(int bits, int hidden, int inter, int K, int has_shared, int sms, int block,
                                    int64_t* out, int n) {
  if (out == nullptr || n < 1 + 8 * kMaxPieces) return FMOE_ERR_INVALID_ARG;
  if ((bits != 4 && bits != 2) || hidden <= 0 || inter <= 0 || hidden % kGroup || inter % kGroup || K < 1 ||
      (has_shared != 0 && has_shared != 1) || sms < 1 || block < 0 || block >= sms)
    return FMOE_ERR_INVALID_ARG;
  const BlobLayout lay = blob_layout(bits, hidden, inter);
  Piece pc[kMaxPieces];
  int darea = 0;
  const int np = block_pieces(K + has_shared, inter, has_shared, block, sms, lay, pc, kMaxPieces, darea);
  for (int i = 0; i < 1 + 8 * kMaxPieces; ++i) out[i] = 0;
  out[0] = np;
  for (int q = 0; q < np && q < kMaxPieces; ++q) {
    const int64_t v[8] = {pc[q].slot, pc[q].i0, pc[q].cnt, pc[q].loc, pc[q].col_off, pc[q].sb_off, pc[q].g0, pc[q].ng};
    for (int k = 0; k < 8; ++k) out[1 + 8 * q + k] = v[k];
  }
  return FMOE_OK;
}

const char* fmoe_status_string(fmoe_status s) {
  switch (s) {
    case FMOE_OK: return "ok";
    case FMOE_ERR_INVALID_ARG: return "invalid argument";
    case FMOE_ERR_UNSUPPORTED: return "unsupported shape or format";
    case FMOE_ERR_CUDA: return "CUDA launch or runtime error";
    case FMOE_ERR_TIMEOUT: return "device-side wait timed out";
    case FMOE_ERR_RANGE: return "a partial output sum exceeded the fixed-point range (|v| > 2^19)";
  }
  return "unknown status";
}

fmoe_status fmoe_last_device_error(void* ws, void* stream) {
  if (ws == nullptr || !aligned(ws, 256)) return FMOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t word = 0;
  cudaError_t e = cudaMemcpyAsync(&word, ws, sizeof(word), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return from_cuda(e);
  if (word != 0) {
    e = cudaMemsetAsync(ws, 0, sizeof(word), st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return from_cuda(e);
  }
  if (word & (kErrWaitTimeout | kErrCopyTimeout)) return FMOE_ERR_TIMEOUT;
  if (word & kErrBadExpert) return FMOE_ERR_INVALID_ARG;
  if (word & kErrRange) return FMOE_ERR_RANGE;
  return FMOE_OK;
}

fmoe_status fmoe_debug_wait_test(void* ws, int n_blocks, int expected, int timeout_us, void* stream) {
  if (ws == nullptr || !aligned(ws, 256)) return FMOE_ERR_INVALID_ARG;
  if (n_blocks < 1 || n_blocks > 148 * 4 || expected < 1 || timeout_us < 1 || timeout_us > 10 * 1000 * 1000)
    return FMOE_ERR_INVALID_ARG;
  uint8_t* base = static_cast<uint8_t*>(ws);
  uint32_t* err = reinterpret_cast<uint32_t*>(base);
  uint32_t* ctr = reinterpret_cast<uint32_t*>(base + 64);   // inside the 256-byte header
  return from_cuda(launch_wait_test(ctr, err, n_blocks, expected, (unsigned long long)timeout_us * 1000ull,
                                    static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
