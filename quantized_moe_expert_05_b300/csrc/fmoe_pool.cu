// Expert slot pool: a fixed number of HBM slots, one expert blob each, filled
// from a copy of every expert in pinned host memory.
//
// The write-ups stream only the K active experts of each layer (~6.75 MB
// each) from SSD and let the OS page cache keep the popular ones (flash-moe
// write-up, discuss.pytorch.kr, section "SSD expert streaming and 'Trust the
// OS'"); the slotstream write-up (simpler24.com) reads experts into a fixed
// pool of slots and evicts unused ones, with whole-expert reads because small
// pieces are far slower ("10 of 512 experts per layer", "the disk was not the
// slow part").  Here host memory stands in for the SSD and HBM slots for the
// page cache: a request (the experts one routing step needs) is planned on
// the host with least-recently-used eviction, each miss is one whole-blob
// cudaMemcpyAsync on a copy stream, and the block then runs against the slot
// pool with router logits remapped to slots.
//
// Everything here is host code; the pool's bookkeeping lives in memory the
// caller provides (fmoe_pool_state_bytes), like the device slots and the
// pinned host blobs.
#include <cfloat>
#include <cstring>

#include "fmoe_kernels.cuh"

namespace {

constexpr uint32_t kPoolMagic = 0x504d4f46u;   // "FOMP"

struct PoolHead {
  uint32_t magic;
  int32_t n_slots, n_experts, pad;
  uint64_t blob_bytes;
  uint64_t tick;           // requests planned so far
  uint64_t hits, misses;   // distinct experts of a request found resident / loaded
  uint8_t* slots_dev;
  const uint8_t* host_blobs;
};

// [head][slot_of: int32 E][expert_of: int32 S][last_use: uint64 S], 8-byte aligned parts
struct PoolView {
  PoolHead* h;
  int32_t* slot_of;
  int32_t* expert_of;
  uint64_t* last_use;
};

size_t round8(size_t v) { return (v + 7) / 8 * 8; }

size_t state_bytes(int S, int E) {
  return round8(sizeof(PoolHead)) + round8((size_t)E * 4) + round8((size_t)S * 4) + (size_t)S * 8;
}

PoolView view(void* state) {
  uint8_t* p = static_cast<uint8_t*>(state);
  PoolView v;
  v.h = reinterpret_cast<PoolHead*>(p);
  const int S = v.h->n_slots, E = v.h->n_experts;
  p += round8(sizeof(PoolHead));
  v.slot_of = reinterpret_cast<int32_t*>(p);
  p += round8((size_t)E * 4);
  v.expert_of = reinterpret_cast<int32_t*>(p);
  p += round8((size_t)S * 4);
  v.last_use = reinterpret_cast<uint64_t*>(p);
  return v;
}

bool valid(const void* state) {
  return state != nullptr && (reinterpret_cast<uintptr_t>(state) % 8) == 0 &&
         static_cast<const PoolHead*>(state)->magic == kPoolMagic;
}

}  // namespace

extern "C" {

size_t fmoe_pool_state_bytes(int n_slots, int n_experts) {
  if (n_slots < 1 || n_experts < 1 || n_experts > FMOE_MAX_EXPERTS) return 0;
  return state_bytes(n_slots, n_experts);
}

fmoe_status fmoe_pool_init(void* state, size_t bytes, int n_slots, int n_experts, size_t blob_bytes, void* slots_dev,
                           const void* host_blobs) {
  if (state == nullptr || (reinterpret_cast<uintptr_t>(state) % 8) != 0) return FMOE_ERR_INVALID_ARG;
  if (n_slots < 1 || n_experts < 1 || n_experts > FMOE_MAX_EXPERTS || bytes < state_bytes(n_slots, n_experts))
    return FMOE_ERR_INVALID_ARG;
  if (blob_bytes == 0 || blob_bytes % 256 != 0 || slots_dev == nullptr || host_blobs == nullptr ||
      (reinterpret_cast<uintptr_t>(slots_dev) % 256) != 0)
    return FMOE_ERR_INVALID_ARG;
  std::memset(state, 0, state_bytes(n_slots, n_experts));
  PoolHead* h = static_cast<PoolHead*>(state);
  h->magic = kPoolMagic;
  h->n_slots = n_slots;
  h->n_experts = n_experts;
  h->blob_bytes = blob_bytes;
  h->slots_dev = static_cast<uint8_t*>(slots_dev);
  h->host_blobs = static_cast<const uint8_t*>(host_blobs);
  PoolView v = view(state);
  for (int e = 0; e < n_experts; ++e) v.slot_of[e] = -1;
  for (int s = 0; s < n_slots; ++s) v.expert_of[s] = -1;
  return FMOE_OK;
}

fmoe_status fmoe_pool_plan(void* state, const int32_t* ids, int n, int keep, int32_t* slots, int32_t* loads,
                           int* n_loads) {
  if (!valid(state) || ids == nullptr || slots == nullptr || loads == nullptr || n_loads == nullptr || n < 1 ||
      keep < 0)
    return FMOE_ERR_INVALID_ARG;
  PoolView v = view(state);
  const int S = v.h->n_slots, E = v.h->n_experts;
  for (int i = 0; i < n; ++i)
    if (ids[i] < 0 || ids[i] >= E) return FMOE_ERR_INVALID_ARG;
  const uint64_t now = v.h->tick + 1;
  // a slot is protected if this request or one of the `keep` before it used it
  const uint64_t protect_from = now > (uint64_t)keep ? now - (uint64_t)keep : 1;
  // capacity first, so that a refused request changes nothing: the distinct
  // missing experts need as many slots that are empty or unprotected and not
  // holding one of the request's resident experts
  int missing = 0;
  for (int i = 0; i < n; ++i) {
    bool first = true;
    for (int j = 0; j < i; ++j) first = first && ids[j] != ids[i];
    if (first && v.slot_of[ids[i]] < 0) ++missing;
  }
  int free_slots = 0;
  for (int c = 0; c < S && free_slots < missing; ++c) {
    if (v.expert_of[c] >= 0 && v.last_use[c] >= protect_from) continue;
    bool used = false;
    for (int i = 0; i < n && !used; ++i) used = v.slot_of[ids[i]] == c;
    if (!used) ++free_slots;
  }
  if (free_slots < missing) return FMOE_ERR_INVALID_ARG;
  v.h->tick = now;
  // resident experts of the request first, so that no miss evicts one of them
  for (int i = 0; i < n; ++i) {
    const int s = v.slot_of[ids[i]];
    if (s >= 0) {
      if (v.last_use[s] != now) ++v.h->hits;
      v.last_use[s] = now;
    }
  }
  int nl = 0;
  for (int i = 0; i < n; ++i) {
    const int e = ids[i];
    int s = v.slot_of[e];
    if (s < 0) {
      // least recently used unprotected slot (an empty slot first; ties to the lower index)
      int best = -1;
      for (int c = 0; c < S; ++c) {
        if (v.expert_of[c] >= 0 && v.last_use[c] >= protect_from) continue;
        const uint64_t key = v.expert_of[c] < 0 ? 0 : v.last_use[c];
        if (best < 0 || key < (v.expert_of[best] < 0 ? 0 : v.last_use[best])) best = c;
      }
      s = best;   // exists: checked above
      if (v.expert_of[s] >= 0) v.slot_of[v.expert_of[s]] = -1;
      v.expert_of[s] = e;
      v.slot_of[e] = s;
      v.last_use[s] = now;
      loads[2 * nl] = e;
      loads[2 * nl + 1] = s;
      ++nl;
      ++v.h->misses;
    }
    slots[i] = s;
  }
  *n_loads = nl;
  return FMOE_OK;
}

fmoe_status fmoe_pool_load(void* state, const int32_t* loads, int n_loads, void* stream) {
  if (!valid(state) || n_loads < 0 || (n_loads > 0 && loads == nullptr)) return FMOE_ERR_INVALID_ARG;
  PoolView v = view(state);
  const size_t b = v.h->blob_bytes;
  for (int i = 0; i < n_loads; ++i) {
    const int e = loads[2 * i], s = loads[2 * i + 1];
    if (e < 0 || e >= v.h->n_experts || s < 0 || s >= v.h->n_slots) return FMOE_ERR_INVALID_ARG;
  }
  for (int i = 0; i < n_loads; ++i) {
    const int e = loads[2 * i], s = loads[2 * i + 1];
    const cudaError_t r = cudaMemcpyAsync(v.h->slots_dev + (size_t)s * b, v.h->host_blobs + (size_t)e * b, b,
                                          cudaMemcpyHostToDevice, static_cast<cudaStream_t>(stream));
    if (r != cudaSuccess) {
      cudaGetLastError();
      return FMOE_ERR_CUDA;
    }
  }
  return FMOE_OK;
}

fmoe_status fmoe_pool_slot_logits(const void* state, const float* logits, const int32_t* ids, const int32_t* slots,
                                  int T, int K, float* slot_logits) {
  if (!valid(state) || logits == nullptr || ids == nullptr || slots == nullptr || slot_logits == nullptr || T < 1 ||
      K < 1)
    return FMOE_ERR_INVALID_ARG;
  const PoolHead* h = static_cast<const PoolHead*>(state);
  const int S = h->n_slots, E = h->n_experts;
  if (K > S) return FMOE_ERR_INVALID_ARG;
  for (int t = 0; t < T; ++t) {
    float* out = slot_logits + (size_t)t * S;
    for (int s = 0; s < S; ++s) out[s] = -FLT_MAX;
    for (int k = 0; k < K; ++k) {
      const int e = ids[t * K + k], s = slots[t * K + k];
      if (e < 0 || e >= E || s < 0 || s >= S) return FMOE_ERR_INVALID_ARG;
      out[s] = logits[(size_t)t * E + e];
    }
  }
  return FMOE_OK;
}

fmoe_status fmoe_pool_stats(const void* state, uint64_t* hits, uint64_t* misses, uint64_t* requests) {
  if (!valid(state)) return FMOE_ERR_INVALID_ARG;
  const PoolHead* h = static_cast<const PoolHead*>(state);
  if (hits != nullptr) *hits = h->hits;
  if (misses != nullptr) *misses = h->misses;
  if (requests != nullptr) *requests = h->tick;
  return FMOE_OK;
}

}  // extern "C"
