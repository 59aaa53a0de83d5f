// Single-launch persistent kernel for batch-1 MoE blocks and stacks of them.
//
// flash-moe (discuss.pytorch.kr write-up, "per-layer pipeline" and "deferred
// CMD3") runs routing, the expert forward and the combine + residual + norm
// per layer as GPU command buffers submitted without waiting; the slotstream
// write-up (simpler24.com, "the disk was not the slow part") measured batch-1
// quantised matmuls at 20 % of memory bandwidth because of dispatch cost.
// Here one cooperative launch (one block per SM) runs every layer.  Block c
// owns intermediate rows [I*c/n, I*(c+1)/n) and output rows [H*c/n, H*(c+1)/n)
// of every selected expert ("slot"); its warps have fixed roles:
//
//   producer       one lane issues every bulk asynchronous copy (TMA engine,
//                  mbarrier completion) of the block's packed rows in the
//                  order they are consumed: gate/up records through a ring
//                  of stages, each slot's down records into its own area.
//                  The shared expert needs no routing, so its rows go first.
//   12 gate/up     dequantised gate/up dot products of the ring's stages
//   warps          against the layer input (pre-scaled, in shared memory);
//                  partial sums per row; a stage is released through an
//                  mbarrier, never a block barrier.
//   finaliser      h = silu(gate) * up for the block's rows, published to L2
//   2 exchange     gather each slot's full h from L2 into shared memory,
//   warps          pre-scaled for the down projection (even / odd slots); the
//                  second also routes: it computes the next layer's top-K at
//                  the end of the current layer and publishes the ids once
//                  that layer's input is complete.
//   4 down warps   fold w_slot * (down_row . h_slot) into per-row sums as each
//                  slot's h arrives; finally out[j] = residual[j] + sum.
//
// Blocks exchange data without counters or barriers: every value published
// to another block (h rows, and the layer outputs of a stack) is stored as
// one 64-bit (value, tag) word whose tag names the launch and layer, so a
// reader knows a value is current from the load that fetches it (the
// low-latency protocol idea of NCCL's LL transport).  A layer's routed
// experts are requested only once its input is complete (their ids are
// published then); the shared expert, which needs no routing, may be
// requested as soon as this block has finished the previous layer.  Every wait is bounded (%globaltimer); a wait
// that runs out records the time-out in the workspace error word, and every
// later wait of the block returns at once, so the launch always ends.
#include "fmoe_async.cuh"
#include "fmoe_kernels.cuh"

namespace fmoe {

namespace {

// (value, tag) words: a float and the tag of the launch and layer that wrote
// it, stored and loaded as one 64-bit access so that a reader sees either the
// old pair or the new one, never a mix.
__device__ __forceinline__ void ll_store(unsigned long long* p, float v, uint32_t tag) {
  const unsigned long long w = ((unsigned long long)tag << 32) | __float_as_uint(v);
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(w) : "memory");
}

__device__ __forceinline__ void ll_load2(const unsigned long long* p, unsigned long long& a, unsigned long long& b) {
  asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
}

__device__ __forceinline__ float ll_value(unsigned long long w) { return __uint_as_float((uint32_t)w); }
__device__ __forceinline__ bool ll_is(unsigned long long w, uint32_t tag) { return (uint32_t)(w >> 32) == tag; }

// Eight consecutive (value, tag) words (16-byte aligned) once all carry
// `tag` (one thread, bounded wait).
__device__ __forceinline__ void ll_wait8(const unsigned long long* p, uint32_t tag, float4& v0, float4& v1,
                                         unsigned long long timeout_ns, uint32_t* err, volatile int* abort) {
  uint64_t t0 = 0;
  bool started = false;
  while (true) {
    unsigned long long w[8];
#pragma unroll
    for (int i = 0; i < 8; i += 2) ll_load2(p + i, w[i], w[i + 1]);
    bool ok = true;
#pragma unroll
    for (int i = 0; i < 8; ++i) ok = ok && ll_is(w[i], tag);
    v0 = make_float4(ll_value(w[0]), ll_value(w[1]), ll_value(w[2]), ll_value(w[3]));
    v1 = make_float4(ll_value(w[4]), ll_value(w[5]), ll_value(w[6]), ll_value(w[7]));
    if (ok || *abort) return;
    const uint64_t t = global_timer_ns();
    if (!started) {
      t0 = t;
      started = true;
    } else if (t - t0 > timeout_ns) {
      atomicOr(err, kErrWaitTimeout);
      *abort = 1;
      return;
    }
    __nanosleep(kInputPollNs);
  }
}

// 16-byte global -> shared copy that holds no registers (completion by
// cp.async.wait_all).  Each 8-byte (value, tag) word of the pair is copied
// whole: an aligned 16-byte read returns every 8-byte half as it was at one
// time.
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Block-wide barrier.  The warps of this kernel take different paths and
// reach it after divergent code (a lane running a loop alone, a row owner
// storing); each warp first reconverges all of its lanes, so that the barrier
// counts whole warps that arrive once each.
__device__ __forceinline__ void cta_sync() {
  __syncwarp();
  asm volatile("barrier.sync 0;" ::: "memory");
}

// named barrier over the consumer warps only (reconverged, as above)
__device__ __forceinline__ void consumer_sync() {
  __syncwarp();
  asm volatile("barrier.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
}

// Reduce four values over `width` consecutive lanes (a power of two, 4..32)
// with a transposed butterfly: on return the group's lane 0 holds sum(a),
// lane width/4 sum(b), lane width/2 sum(c) and lane 3*width/4 sum(d).
__device__ __forceinline__ float quad_reduce(float a, float b, float c, float d, int width, int lane) {
  const int half = width >> 1, quarter = width >> 2;
  const bool lo = (lane & half) == 0;
  const float s0 = __shfl_xor_sync(0xFFFFFFFFu, lo ? c : a, half);
  const float s1 = __shfl_xor_sync(0xFFFFFFFFu, lo ? d : b, half);
  const float x0 = (lo ? a : c) + s0;
  const float x1 = (lo ? b : d) + s1;
  const bool lq = (lane & quarter) == 0;
  float y = (lq ? x0 : x1) + __shfl_xor_sync(0xFFFFFFFFu, lq ? x1 : x0, quarter);
  for (int o = quarter >> 1; o >= 1; o >>= 1) y += __shfl_xor_sync(0xFFFFFFFFu, y, o);
  return y;
}

}  // namespace

// Slice s of a slot's staged h (float4 j of slice s at j*hstride + s, already
// pre-scaled): the 32 values as pairs, and their plain sum, taken from the
// pre-scaled values one position class at a time (an exact power-of-two
// rescaling each).
template <int BITS>
__device__ __forceinline__ float staged_h_slice(const float4* hs4, int hstride, int s, SliceX& hs) {
  float2 c01 = make_float2(0.f, 0.f), c23 = make_float2(0.f, 0.f);
  float2 c45 = make_float2(0.f, 0.f), c67 = make_float2(0.f, 0.f);
#pragma unroll
  for (int j = 0; j < kSlice / 4; ++j) {
    const float4 v = hs4[(size_t)j * hstride + s];
    hs[2 * j] = make_float2(v.x, v.y);
    hs[2 * j + 1] = make_float2(v.z, v.w);
    if (BITS == 4 || (j & 1) == 0) {
      c01 = __fadd2_rn(c01, hs[2 * j]);
      c23 = __fadd2_rn(c23, hs[2 * j + 1]);
    } else {
      c45 = __fadd2_rn(c45, hs[2 * j]);
      c67 = __fadd2_rn(c67, hs[2 * j + 1]);
    }
  }
  float hsm = (c01.x * inv_pos_scale<BITS>(0) + c01.y * inv_pos_scale<BITS>(1)) +
              (c23.x * inv_pos_scale<BITS>(2) + c23.y * inv_pos_scale<BITS>(3));
  if (BITS == 2)
    hsm += (c45.x * inv_pos_scale<BITS>(4) + c45.y * inv_pos_scale<BITS>(5)) +
           (c67.x * inv_pos_scale<BITS>(6) + c67.y * inv_pos_scale<BITS>(7));
  return hsm;
}

// w * (down row r . h) over slice s: the row's record in shared memory.
template <int BITS>
__device__ __forceinline__ float down_slice(const uint8_t* rec, const BlobLayout& lay, int s, const SliceX& hs,
                                            float hsm, float w, float acc) {
  SliceCodes<BITS> q;
  if constexpr (BITS == 4) q.v = *reinterpret_cast<const uint4*>(rec + (size_t)s * 16);
  else q.v = *reinterpret_cast<const uint2*>(rec + (size_t)s * 8);
  const uint32_t sbw = *reinterpret_cast<const uint32_t*>(rec + lay.qi + (size_t)(s >> 1) * 4);
  return fmaf(w, slice_term<BITS>(q, sbw, hs, hsm), acc);
}

template <int BITS>
__global__ void __maxnreg__(kFusedMaxRegs) fused_moe_kernel(const __grid_constant__ FusedParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const FusedPlan& pl = p.plan;
  const BlobLayout& lay = p.lay;
  // control area
  uint64_t* bar_full = reinterpret_cast<uint64_t*>(smem);          // ring stage filled (count 1 + bytes)
  uint64_t* bar_empty = bar_full + kMaxStages;                      // ring stage released (one per consumer warp)
  uint64_t* bar_dfull = bar_empty + kMaxStages;                     // slot's down records filled
  uint64_t* bar_routed = bar_dfull + kMaxSlots;                     // slot's expert id known
  uint64_t* bar_slot = bar_routed + kMaxSlots;                      // slot's partial sums written
  uint64_t* bar_hready = bar_slot + kMaxSlots;                      // slot's full h staged
  uint64_t* bar_xready = bar_hready + kMaxSlots;                    // layer input complete (consumers)
  uint64_t* bar_ddone = bar_xready + 1;                             // slot's down records used (down warps)
  uint64_t* bar_layer = bar_ddone + kMaxSlots;                      // layer done (every warp but the producer)
  uint64_t* bar_tail = bar_layer + 1;                               // tail slots' down rows done (gate/up warps)
  float* s_tail = reinterpret_cast<float*>(smem + 1536);            // [nd] tail slots' sum per down row
  int* s_ids = reinterpret_cast<int*>(smem + 1024);                 // [kMaxSlots]
  float* s_w = reinterpret_cast<float*>(smem + 1152);               // [kMaxSlots] routing weights, shared gate
  float* s_red = reinterpret_cast<float*>(smem + 1280);             // [kConsumerWarps][2]
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + 1408);
  float* s_part = reinterpret_cast<float*>(smem + pl.part_off);    // [slot][row][part][2]
  unsigned long long* s_stage = reinterpret_cast<unsigned long long*>(smem + pl.stage_off);  // one slot's h words
  uint8_t* s_hs = smem + pl.hs_off;                                // [slot] h slices + slice sums
  float4* s_x4 = reinterpret_cast<float4*>(smem + pl.xs_off);      // layer input, slice-major
  uint8_t* darea = smem + pl.darea_off;                            // [slot] down records
  uint8_t* ring = smem + pl.ring_off;                              // [stage] gate/up records

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int c = blockIdx.x, n = gridDim.x;
  const int NS = p.K + p.S;
  const int H = p.H, I = p.I;

  // Gate/up: this block owns rows [ra, ra+nr) of every slot.  The rows of
  // all slots form one sequence of NS*nr "virtual rows" (slot-major) that
  // the ring carries R at a time; a gate/up warp handles rows rs0 and rs1
  // of each stage (its slice range `sl` of H).
  const int tl = H / kSlice;
  const int R = pl.rows_per_stage;
  const int nparts = pl.nparts;
  const int gw = tl < 32 ? tl : 32;                                // reduction width
  const int ra = (int)((long long)I * c / n);
  const int nr = (int)((long long)I * (c + 1) / n) - ra;
  const int V = NS * nr;
  const int nstg = (V + R - 1) / R;
  int rs0, sl, pi;
  if (tl >= 32) {
    rs0 = warp < (R / 2) * nparts ? warp / nparts : R;   // warps beyond a whole pass stay idle
    pi = warp % nparts;
    sl = pi * 32 + lane;
  } else {
    rs0 = warp * (32 / tl) + lane / tl;
    pi = 0;
    sl = lane % tl;
  }
  const int rs1 = rs0 + R / 2;
  // Down: this block owns output rows [ja, ja+nd); a row has tld slices;
  // lpr lanes per row, rpp rows per warp pass.  Staged h: float4 j of slice
  // s at j*(tld+1) + s (the padding keeps the exchanger's stores free of
  // bank conflicts), then the tld slice sums.
  const int ja = (int)((long long)H * c / n);
  const int nd = (int)((long long)H * (c + 1) / n) - ja;
  const int tld = I / kSlice;
  const int hstride = tld + 1;
  const int lpr = tld < 32 ? tld : 32;
  const int rpp = 32 / lpr;
  const int spl = tld > 32 ? tld / 32 : 1;
  const int ngroups = (nd + rpp - 1) / rpp;
  const int dlag = pl.dlag;
  // slots whose down rows the gate/up warps take over at the end of a layer
  const int ntail = NS - 1 < kFusedTailSlots ? NS - 1 : kFusedTailSlots;

  if (tid == 0) {
    for (int i = 0; i < kMaxStages; ++i) {
      mbar_init(&bar_full[i], 1);
      mbar_init(&bar_empty[i], kGuWarps);
    }
    for (int i = 0; i < kMaxSlots; ++i) {
      mbar_init(&bar_dfull[i], 1);
      mbar_init(&bar_routed[i], 1);
      mbar_init(&bar_slot[i], kGuWarps);
      mbar_init(&bar_hready[i], 1);
    }
    mbar_init(bar_xready, 1);
    for (int i = 0; i < kMaxSlots; ++i) mbar_init(&bar_ddone[i], kDownWarps);
    mbar_init(bar_layer, kFusedThreads / 32 - 1);
    mbar_init(bar_tail, kGuWarps);
    *s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  cta_sync();

  uint32_t g_issue = 0;   // gate/up stages issued (producer warp)
  uint32_t n_copies = 0;  // bulk copies issued (producer warp): picks the issuing lane
  uint32_t g_cons = 0;    // gate/up stages consumed (consumer warps)
  const unsigned long long tmo = p.timeout_ns;
  // tags of this launch: layer l publishes with epoch * 64 + l + 1 (never 0,
  // the value of a freshly zeroed workspace)
  const uint32_t tag0 = *reinterpret_cast<volatile uint32_t*>(p.epoch) * (uint32_t)kMaxFusedLayers + 1u;

  int nx_id = -1;       // routing exchange warp: top-K pick of its lane for the coming layer
  float nx_l = 0.f;
  for (int l = 0; l < p.L; ++l) {
    const FusedLayerPtrs lp = p.layer[l];
    const uint32_t lpar = (uint32_t)(l & 1);
    const uint32_t tag = tag0 + (uint32_t)l;
    // input: x (block), the stack input h (layer 0), or the previous layer's
    // published output; residual likewise; output: out, or published words
    const bool in_ll = p.norm && l > 0;
    const bool out_ll = p.norm && l < p.L - 1;
    const float* hin = p.norm ? p.out : p.x;
    const unsigned long long* hin_ll = p.hbufll + (size_t)((l - 1) & 1) * H;
    unsigned long long* out_llp = p.hbufll + (size_t)(l & 1) * H;
    // slot ps: 0 is the shared expert when there is one; its h goes to index K
    auto hidx = [&](int ps) -> int { return p.S ? (ps == 0 ? p.K : ps - 1) : ps; };

    if (warp == kProducerWarp) {
      // ------------------------------------------------------------------
      // producer: the warp walks the layer's copies in consumption order;
      // lane 0 declares each barrier's bytes, and successive copies are
      // issued by successive lanes: the copies one thread issues are carried
      // out one after another, those of different threads side by side
      // ------------------------------------------------------------------
#if FMOE_FUSED_LATE_PREFETCH
      // the previous layer's exchanges go first: its last slot's h staged
      if (l > 0) mbar_wait(&bar_hready[NS - 1], (uint32_t)((l - 1) & 1), tmo, p.err, s_abort);
#endif
      auto slot_blob = [&](int ps) -> const uint8_t* {
        if (p.S && ps == 0) return lp.shared;
        return lp.experts + (size_t)s_ids[ps] * p.blob;
      };
      // lane 0's view of the abort flag, the same in every lane
      auto aborted = [&]() -> bool { return __shfl_sync(0xFFFFFFFFu, *s_abort, 0) != 0; };
      bool routed = false;       // routed ids are published all at once
      auto ensure_routed = [&](int ps) {
        if (ps >= p.S && !routed) {
          mbar_wait(&bar_routed[0], lpar, tmo, p.err, s_abort);
          routed = true;
        }
      };
      auto copy = [&](void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
        if (lane == (int)(n_copies % kFusedIssueLanes)) bulk_g2s(dst, src, bytes, bar);
        ++n_copies;
      };
      auto issue_down = [&](int ps) {
        // the previous layer's down work is done with this slot's area
        if (l > 0) mbar_wait(&bar_ddone[ps], (uint32_t)((l - 1) & 1), tmo, p.err, s_abort);
        if (nd == 0 || aborted()) {
          if (lane == 0) mbar_arrive_expect_tx(&bar_dfull[ps], 0);
          return;
        }
        ensure_routed(ps);
        if (lane == 0) mbar_arrive_expect_tx(&bar_dfull[ps], (uint32_t)(nd * lay.d_row));
        __syncwarp();
        const int per = (nd + kFusedDownCopies - 1) / kFusedDownCopies;
        for (int r0 = 0; r0 < nd; r0 += per)
          copy(darea + (size_t)ps * pl.dslot_bytes + (size_t)r0 * lay.d_row,
               slot_blob(ps) + lay.d_off + (size_t)(ja + r0) * lay.d_row, (uint32_t)(min(per, nd - r0) * lay.d_row),
               &bar_dfull[ps]);
      };
      int dnext = 0;
      for (int k = 0; k < nstg; ++k) {
        const uint32_t st = g_issue % pl.nstage;
        const uint32_t use = g_issue / pl.nstage;
        ++g_issue;
        if (use >= 1) mbar_wait(&bar_empty[st], (use - 1) & 1u, tmo, p.err, s_abort);
        const int v0 = k * R, v1 = min(V, v0 + R);
        if (aborted()) {
          if (lane == 0) mbar_arrive_expect_tx(&bar_full[st], 0);
        } else {
          // the stage's bytes are expected up front; the shared expert's
          // segment goes out at once, routed segments once ids are known
          if (lane == 0) mbar_arrive_expect_tx(&bar_full[st], (uint32_t)((v1 - v0) * lay.gu_row));
          __syncwarp();
          uint8_t* buf = ring + (size_t)st * pl.stage_bytes;
          for (int v = v0; v < v1;) {           // copies of at most kFusedRowsPerCopy rows of one slot
            const int ps = v / nr, r = v % nr;
            const int cnt = min(min(v1 - v, nr - r), kFusedRowsPerCopy);
            ensure_routed(ps);
            if (!aborted())
              copy(buf + (size_t)(v - v0) * lay.gu_row, slot_blob(ps) + (size_t)(ra + r) * lay.gu_row,
                   (uint32_t)(cnt * lay.gu_row), &bar_full[st]);
            v += cnt;
          }
        }
        // down records of slots whose gate/up is dlag slots behind
        const int slots_issued = v1 / nr;
        while (dnext < slots_issued - dlag) issue_down(dnext++);
      }
      while (dnext < NS) issue_down(dnext++);
      __syncwarp();
    } else if (warp == kFinalWarp) {
      // ------------------------------------------------------------------
      // finaliser: h = silu(gate . x) * (up . x) for this block's rows, to L2
      // ------------------------------------------------------------------
      for (int ps = 0; ps < NS; ++ps) {
        mbar_wait(&bar_slot[ps], lpar, tmo, p.err, s_abort);
        float* hdst = p.hmid + (size_t)hidx(ps) * I + ra;
        unsigned long long* hll = p.hll + (size_t)hidx(ps) * I + ra;
        const float* part = s_part + (size_t)ps * pl.nrmax * nparts * 2;
        for (int r = lane; r < nr; r += 32) {
          float a = 0.f, u = 0.f;
          for (int q = 0; q < nparts; ++q) {
            a += part[(r * nparts + q) * 2];
            u += part[(r * nparts + q) * 2 + 1];
          }
          const float hv = silu_f(a) * u;
          ll_store(hll + r, hv, tag);
          if (l == p.L - 1) hdst[r] = hv;
        }
      }
    } else if (warp == kExchangeWarp || warp == kExchangeWarp2) {
      // ------------------------------------------------------------------
      // exchangers: each slot's full h from L2 into shared memory, the first
      // exchanger taking even slots, the second odd; the second also routes
      // ------------------------------------------------------------------
      const int xw = warp - kExchangeWarp;
      if (xw == kRouteXw) {
        // the layer's top-K: computed at the end of the previous layer (the
        // logits are inputs), or now for the first layer of the launch
        if (l == 0) warp_topk(p.logits, p.E, p.K, nx_id, nx_l);
        const int my_id = nx_id;
        const float my_w = warp_topk_softmax(nx_l, p.K);
        // publish once the consumers hold the whole layer input
        mbar_wait(bar_xready, lpar, tmo, p.err, s_abort);
        if (lane < p.K) {
          s_ids[p.S + lane] = my_id;
          s_w[p.S + lane] = my_w;
          if (c == 0 && p.ids_out != nullptr) {
            p.ids_out[(size_t)l * p.K + lane] = my_id;
            p.w_out[(size_t)l * p.K + lane] = my_w;
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_routed[0]);
      }
      unsigned long long* my_stage = s_stage + (size_t)xw * I;
      for (int q = xw; q < NS; q += 2) {
        const unsigned long long* hsrc = p.hll + (size_t)hidx(q) * I;
        float* hsf = reinterpret_cast<float*>(s_hs + (size_t)q * pl.hs_slot_bytes);
#if FMOE_XCHG_WAIT_OWN
        // the other blocks finish a slot at about the time this one does:
        // polling earlier only returns stale words one round trip later
        mbar_wait(&bar_slot[q], lpar, tmo, p.err, s_abort);
#endif
        // fetch all I words of the slot, then re-fetch until every tag is current
        uint64_t t0 = 0;
        bool started = false;
        while (true) {
          for (int c2 = lane; c2 < I / 2; c2 += 32) cp_async16(my_stage + 2 * c2, hsrc + 2 * c2);
          cp_async_wait_all();
          __syncwarp();
          bool ok = true;
          for (int i = lane; i < I; i += 32) ok = ok && ll_is(my_stage[i], tag);
          if (__all_sync(0xFFFFFFFFu, ok)) break;
          if (*s_abort) break;
          const uint64_t t = global_timer_ns();
          if (!started) {
            t0 = t;
            started = true;
          } else if (t - t0 > tmo) {
            atomicOr(p.err, kErrWaitTimeout);
            *s_abort = 1;
            break;
          }
          __nanosleep(kExchangePollNs);
        }
        // pre-scale into the padded slice-major layout; lane = position in the
        // slice, so that the reads are consecutive and the stores hit 32 banks
        const float ps_l = pos_scale<BITS>(lane);
        const int fo = ((lane >> 2) * hstride) * 4 + (lane & 3);
#pragma unroll 8
        for (int m = 0; m < tld; ++m) hsf[fo + m * 4] = ll_value(my_stage[(size_t)m * kSlice + lane]) * ps_l;
        __threadfence_block();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_hready[q]);
      }
      // the next layer's top-K, off its critical path; its ids are published
      // only once that layer's input is complete
      if (xw == kRouteXw && l + 1 < p.L) warp_topk(p.logits + (size_t)(l + 1) * p.E, p.E, p.K, nx_id, nx_l);
    } else {
      // ------------------------------------------------------------------
      // consumers: 12 gate/up warps and 4 down warps
      // ------------------------------------------------------------------
      float rinv;
      {
        // The layer input goes through shared memory, slice-major (float4 j of
        // slice s at j*tl + s), so that each lane then reads its slice without
        // bank conflicts.  Every consumer thread fetches 8 consecutive elements
        // (plain, or published words of the previous layer) and adds up their
        // squares and their products with the shared-expert gate vector.
        float ss = 0.f, wg = 0.f;
        for (int e = tid * 8; e < H; e += kConsumerWarps * 32 * 8) {
          float4 v0, v1;
          if (in_ll) {
            ll_wait8(hin_ll + e, tag - 1u, v0, v1, tmo, p.err, s_abort);
          } else {
            const float4* src = reinterpret_cast<const float4*>(hin + e);
            v0 = p.norm ? __ldcg(src) : __ldg(src);
            v1 = p.norm ? __ldcg(src + 1) : __ldg(src + 1);
          }
          s_x4[((e & 31) >> 2) * tl + (e >> 5)] = v0;
          s_x4[(((e + 4) & 31) >> 2) * tl + (e >> 5)] = v1;
          ss += (v0.x * v0.x + v0.y * v0.y) + (v0.z * v0.z + v0.w * v0.w);
          ss += (v1.x * v1.x + v1.y * v1.y) + (v1.z * v1.z + v1.w * v1.w);
          if (p.S) {
            const uint4 wb = __ldg(reinterpret_cast<const uint4*>(lp.wsg + e));
            wg += (bf16lo(wb.x) * v0.x + bf16hi(wb.x) * v0.y) + (bf16lo(wb.y) * v0.z + bf16hi(wb.y) * v0.w);
            wg += (bf16lo(wb.z) * v1.x + bf16hi(wb.z) * v1.y) + (bf16lo(wb.w) * v1.z + bf16hi(wb.w) * v1.w);
          }
        }
        ss = warp_sum(ss);
        wg = warp_sum(wg);
        if (lane == 0) {
          s_red[2 * warp] = ss;
          s_red[2 * warp + 1] = wg;
        }
        consumer_sync();
        float tot = 0.f, wgt = 0.f;
#pragma unroll
        for (int q = 0; q < kConsumerWarps; ++q) {
          tot += s_red[2 * q];
          wgt += s_red[2 * q + 1];
        }
        rinv = p.norm ? 1.0f / sqrtf(tot / (float)H + p.eps) : 1.0f;
        if (warp == 0 && lane == 0) {
          const float gate = p.S ? sigmoid_f(wgt * rinv) : 0.f;
          if (p.S) s_w[0] = gate;
          if (c == 0 && p.gate_out != nullptr) p.gate_out[l] = gate;
          mbar_arrive(bar_xready);
        }
      }

      if (warp < kGuWarps) {
        // ---------------- gate/up: stream the ring, partial sums to smem ----
        SliceX xs;
        float xsum = 0.f;
#pragma unroll
        for (int j = 0; j < kSlice / 4; ++j) {
          const float4 v = s_x4[j * tl + sl];
          xsum += put_x4<BITS>(xs, j, make_float4(v.x * rinv, v.y * rinv, v.z * rinv, v.w * rinv));
        }
        int next_done = 0;
        if (nr == 0) {               // no gate/up rows here: every slot is complete at once
          __syncwarp();
          if (lane == 0)
            for (int ps = 0; ps < NS; ++ps) mbar_arrive(&bar_slot[ps]);
          next_done = NS;
        }
        for (int k = 0; k < nstg; ++k) {
          const uint32_t st = g_cons % pl.nstage;
          mbar_wait(&bar_full[st], (g_cons / pl.nstage) & 1u, tmo, p.err, s_abort);
          ++g_cons;
          const uint8_t* buf = ring + (size_t)st * pl.stage_bytes;
          const int v0 = k * R + rs0, v1 = k * R + rs1;
          float ga0 = 0.f, ua0 = 0.f, ga1 = 0.f, ua1 = 0.f;
          if (rs0 < R / 2 && v0 < V) {
            const uint8_t* rec = buf + (size_t)rs0 * lay.gu_row;
            SliceCodes<BITS> qg, qu;
            if constexpr (BITS == 4) {
              qg.v = *reinterpret_cast<const uint4*>(rec + (size_t)sl * 16);
              qu.v = *reinterpret_cast<const uint4*>(rec + lay.qh + (size_t)sl * 16);
            } else {
              qg.v = *reinterpret_cast<const uint2*>(rec + (size_t)sl * 8);
              qu.v = *reinterpret_cast<const uint2*>(rec + lay.qh + (size_t)sl * 8);
            }
            const uint32_t sg = *reinterpret_cast<const uint32_t*>(rec + 2 * lay.qh + (size_t)(sl >> 1) * 4);
            const uint32_t su = *reinterpret_cast<const uint32_t*>(rec + 2 * lay.qh + lay.sh + (size_t)(sl >> 1) * 4);
            ga0 = slice_term<BITS>(qg, sg, xs, xsum);
            ua0 = slice_term<BITS>(qu, su, xs, xsum);
          }
          if (rs0 < R / 2 && v1 < V) {
            const uint8_t* rec = buf + (size_t)rs1 * lay.gu_row;
            SliceCodes<BITS> qg, qu;
            if constexpr (BITS == 4) {
              qg.v = *reinterpret_cast<const uint4*>(rec + (size_t)sl * 16);
              qu.v = *reinterpret_cast<const uint4*>(rec + lay.qh + (size_t)sl * 16);
            } else {
              qg.v = *reinterpret_cast<const uint2*>(rec + (size_t)sl * 8);
              qu.v = *reinterpret_cast<const uint2*>(rec + lay.qh + (size_t)sl * 8);
            }
            const uint32_t sg = *reinterpret_cast<const uint32_t*>(rec + 2 * lay.qh + (size_t)(sl >> 1) * 4);
            const uint32_t su = *reinterpret_cast<const uint32_t*>(rec + 2 * lay.qh + lay.sh + (size_t)(sl >> 1) * 4);
            ga1 = slice_term<BITS>(qg, sg, xs, xsum);
            ua1 = slice_term<BITS>(qu, su, xs, xsum);
          }
          const float v = quad_reduce(ga0, ua0, ga1, ua1, gw, lane);
          const int pos = lane & (gw - 1), qw = gw >> 2;
          const int vv = pos < 2 * qw ? v0 : v1;
          if (rs0 < R / 2 && vv < V && (pos & (qw - 1)) == 0) {
            const int ps = vv / nr, r = vv % nr;
            s_part[(((size_t)ps * pl.nrmax + r) * nparts + pi) * 2 + ((pos / qw) & 1)] = v;
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&bar_empty[st]);
          // slots whose last row was in this stage are complete
          const int last_v = min(V, (k + 1) * R);
          bool fenced = false;
          while (next_done < NS && (next_done + 1) * nr <= last_v) {
            if (!fenced) {
              __threadfence_block();
              __syncwarp();
              fenced = true;
            }
            if (lane == 0) mbar_arrive(&bar_slot[next_done]);
            ++next_done;
          }
        }
        if (ntail > 0) {
          // the last slots' down rows: by the time their h is gathered the
          // gate/up warps are idle, and twelve warps finish a slot sooner
          // than the four down warps, whose every instruction waits on the
          // one before it
          float tacc[kMaxTailGroups];
#pragma unroll
          for (int gi = 0; gi < kMaxTailGroups; ++gi) tacc[gi] = 0.f;
          for (int ps = NS - ntail; ps < NS; ++ps) {
            mbar_wait(&bar_hready[ps], lpar, tmo, p.err, s_abort);
            mbar_wait(&bar_dfull[ps], lpar, tmo, p.err, s_abort);
            const float wk = s_w[ps];
            const float4* hs4 = reinterpret_cast<const float4*>(s_hs + (size_t)ps * pl.hs_slot_bytes);
            const uint8_t* buf = darea + (size_t)ps * pl.dslot_bytes;
            for (int k = 0; k < spl; ++k) {
              const int s = (lane % lpr) + 32 * k;
              SliceX hs;
              const float hsm = staged_h_slice<BITS>(hs4, hstride, s, hs);
#pragma unroll
              for (int gi = 0; gi < kMaxTailGroups; ++gi) {
                const int grp = warp + kGuWarps * gi;
                const int r = grp * rpp + lane / lpr;
                if (grp < ngroups && r < nd)
                  tacc[gi] = down_slice<BITS>(buf + (size_t)r * lay.d_row, lay, s, hs, hsm, wk, tacc[gi]);
              }
            }
          }
#pragma unroll
          for (int gi = 0; gi < kMaxTailGroups; ++gi) {
            const int grp = warp + kGuWarps * gi;
            const float v = warp_sum(tacc[gi], lpr);
            const int r = grp * rpp + lane / lpr;
            if (grp < ngroups && r < nd && (lane % lpr) == 0) s_tail[r] = v;
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_tail);
        }
      } else {
        // ---------------- down projection + combine + residual -------------
        const int dw = warp - kGuWarps;
        float acc[kMaxDownGroups];
        float resv[kMaxDownGroups];
#pragma unroll
        for (int gi = 0; gi < kMaxDownGroups; ++gi) {
          const int grp = dw + kDownWarps * gi;
          const int r = grp * rpp + lane / lpr;
          acc[gi] = 0.f;
          resv[gi] = 0.f;
          if (grp < ngroups && r < nd && (lane % lpr) == 0) {
            if (p.norm) {
              const int e = ja + r;
              resv[gi] = reinterpret_cast<const float*>(s_x4)[(((e & 31) >> 2) * tl + (e >> 5)) * 4 + (e & 3)];
            } else {
              resv[gi] = __ldg(p.residual + ja + r);
            }
          }
        }
        for (int ps = 0; ps < NS - ntail; ++ps) {
          mbar_wait(&bar_hready[ps], lpar, tmo, p.err, s_abort);
          mbar_wait(&bar_dfull[ps], lpar, tmo, p.err, s_abort);
          const float wk = s_w[ps];
          const float4* hs4 = reinterpret_cast<const float4*>(s_hs + (size_t)ps * pl.hs_slot_bytes);
          const uint8_t* buf = darea + (size_t)ps * pl.dslot_bytes;
          for (int k = 0; k < spl; ++k) {
            const int s = (lane % lpr) + 32 * k;
            SliceX hs;
            const float hsm = staged_h_slice<BITS>(hs4, hstride, s, hs);
#pragma unroll
            for (int gi = 0; gi < kMaxDownGroups; ++gi) {
              const int grp = dw + kDownWarps * gi;
              const int r = grp * rpp + lane / lpr;
              if (grp < ngroups && r < nd)
                acc[gi] = down_slice<BITS>(buf + (size_t)r * lay.d_row, lay, s, hs, hsm, wk, acc[gi]);
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&bar_ddone[ps]);
        }
        if (ntail > 0) {
          // the tail slots' rows were done by the gate/up warps
          mbar_wait(bar_tail, lpar, tmo, p.err, s_abort);
          __syncwarp();
          if (lane == 0)
            for (int ps = NS - ntail; ps < NS; ++ps) mbar_arrive(&bar_ddone[ps]);
        }
        // combine + residual, written by each row's owner
#pragma unroll
        for (int gi = 0; gi < kMaxDownGroups; ++gi) {
          const int grp = dw + kDownWarps * gi;
          const float v = warp_sum(acc[gi], lpr);
          const int r = grp * rpp + lane / lpr;
          if (grp < ngroups && r < nd && (lane % lpr) == 0) {
            const float o = resv[gi] + v + (ntail > 0 ? s_tail[r] : 0.f);
            if (out_ll) ll_store(out_llp + ja + r, o, tag);
            else p.out[ja + r] = o;
          }
        }
      }
    }

    // ---- end of layer: every role but the producer is done with this
    // layer's shared memory.  The producer runs on into the next layer: the
    // ring's stages come back to it through bar_empty and the down areas
    // through bar_ddone, so it may request the next layer's shared expert
    // while this layer's down projection finishes.
    if (warp != kProducerWarp) {
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_layer);
      mbar_wait(bar_layer, lpar, tmo, p.err, s_abort);
    }
  }

  // No copy may still be writing this block's shared memory when it exits:
  // wait (bounded, whether or not the block gave up) for the last phase of
  // every stage and down area that was used.
  if (warp == kProducerWarp && lane == 0) {
    volatile int no_abort = 0;
    const uint32_t used = g_issue < (uint32_t)pl.nstage ? g_issue : (uint32_t)pl.nstage;
    for (uint32_t st = 0; st < used; ++st) {
      const uint32_t last = g_issue - 1 - ((g_issue - 1 - st) % pl.nstage);   // last issue index of stage st
      mbar_wait(&bar_full[st], (last / pl.nstage) & 1u, tmo, p.err, &no_abort);
    }
    for (int ps = 0; ps < NS; ++ps) mbar_wait(&bar_dfull[ps], (uint32_t)((p.L - 1) & 1), tmo, p.err, &no_abort);
  }

  // the last block out starts the next epoch of tags and resets the exit count
  cta_sync();
  if (tid == 0) {
    __threadfence();
    const uint32_t old = atomicAdd(p.exit_ctr, 1u);
    if (old == (uint32_t)n - 1) {
      *p.exit_ctr = 0;
      atomicAdd(p.epoch, 1u);
      __threadfence();
    }
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
static bool pow2(int v) { return v > 0 && (v & (v - 1)) == 0; }
static int round_up_i(long long v, int a) { return (int)((v + a - 1) / a * a); }

FusedPlan fused_plan(int bits, int H, int I, int K, int S, int device) {
  int sms = 0, smem_max = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess ||
      cudaDeviceGetAttribute(&smem_max, cudaDevAttrMaxSharedMemoryPerBlockOptin, device) != cudaSuccess) {
    cudaGetLastError();
    FusedPlan pl{};
    pl.ok = false;
    return pl;
  }
  return fused_plan_for(bits, H, I, K, S, sms, smem_max);
}

FusedPlan fused_plan_for(int bits, int H, int I, int K, int S, int sms, int smem_max) {
  FusedPlan pl{};
  pl.ok = false;
  const int tl = H / kSlice, tld = I / kSlice;
  if (H % kSlice || I % kSlice || !pow2(tl) || !pow2(tld)) return pl;
  if (tl < 4 || tl > 32 * kConsumerWarps || tld < 1) return pl;
  if (K + S > kMaxSlots || K < 1 || sms < 1) return pl;
  const int grid = sms;
  const int NS = K + S;
  const BlobLayout lay = blob_layout(bits, H, I);
  // gate/up stage: two rows per consumer warp and slice range
  const int nparts = tl >= 32 ? tl / 32 : 1;
  if (nparts > kGuWarps) return pl;
  const int R = 2 * (tl >= 32 ? kGuWarps / nparts : kGuWarps * (32 / tl));
  pl.rows_per_stage = R;
  pl.nparts = nparts;
  pl.stage_bytes = round_up_i((long long)R * lay.gu_row, 128);
  // down records of one slot
  const int ndmax = (H + grid - 1) / grid;
  const int lpr = tld < 32 ? tld : 32, rpp = 32 / lpr;
  if ((ndmax + rpp - 1) / rpp > kMaxDownGroups * kDownWarps) return pl;
  if ((ndmax + rpp - 1) / rpp > kMaxTailGroups * kGuWarps || ndmax > kMaxTailRows) return pl;
  pl.dslot_bytes = round_up_i((long long)ndmax * lay.d_row, 128);
  pl.nrmax = (I + grid - 1) / grid;
  pl.hs_slot_bytes = round_up_i((long long)8 * (tld + 1) * 16, 128);
  pl.part_off = kCtrlBytes;
  pl.stage_off = round_up_i(pl.part_off + (long long)NS * pl.nrmax * nparts * 2 * 4, 128);
  pl.hs_off = round_up_i(pl.stage_off + (long long)2 * I * 8, 128);
  // the layer input is staged where the slots' h will go: it is read by the
  // consumers before their first gate/up stage, and the first h is written
  // only after every block has finished a slot
  pl.xs_off = pl.hs_off;
  const long long hs_region = (long long)NS * pl.hs_slot_bytes > (long long)H * 4 ? (long long)NS * pl.hs_slot_bytes
                                                                                  : (long long)H * 4;
  pl.darea_off = round_up_i(pl.hs_off + hs_region, 128);
  pl.ring_off = pl.darea_off + NS * pl.dslot_bytes;
  const long long avail = (long long)smem_max - pl.ring_off;
  const long long ns = avail / pl.stage_bytes;
  if (ns < 2) return pl;
  pl.nstage = (int)(ns > kFusedStageCap ? kFusedStageCap : ns);
  pl.smem = (size_t)pl.ring_off + (size_t)pl.nstage * pl.stage_bytes;
  pl.dlag = kFusedDownLag;
  pl.grid = grid;
  pl.ok = true;
  return pl;
}

template <int BITS>
static cudaError_t launch_fused_t(FusedParams& p, const FusedPlan& pl, cudaStream_t st) {
  // the shared-memory limit and the residency check, once per device and size
  // (function attributes belong to the device's context)
  static int configured_smem[64];
  static size_t checked_smem[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (configured_smem[dev] < (int)pl.smem) {
    e = cudaFuncSetAttribute(fused_moe_kernel<BITS>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pl.smem);
    if (e != cudaSuccess) return e;
    configured_smem[dev] = (int)pl.smem;
  }
  if (checked_smem[dev] != pl.smem) {
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fused_moe_kernel<BITS>, kFusedThreads, pl.smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorCooperativeLaunchTooLarge;
    checked_smem[dev] = pl.smem;
  }
  // cooperative: all blocks resident at once (every block waits for words
  // that the other blocks publish)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(pl.grid);
  cfg.blockDim = dim3(kFusedThreads);
  cfg.dynamicSmemBytes = pl.smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fused_moe_kernel<BITS>, p);
}

cudaError_t launch_fused(FusedParams& p, const FusedPlan& pl, cudaStream_t st) {
  p.plan = pl;
  return p.bits == 4 ? launch_fused_t<4>(p, pl, st) : launch_fused_t<2>(p, pl, st);
}

// ---------------------------------------------------------------------------
// bounded-wait test kernel: every block arrives once, then waits for
// `expected` arrivals; the last block out resets the counter.
// ---------------------------------------------------------------------------
__global__ void wait_test_kernel(uint32_t* counter, uint32_t* err, int expected, unsigned long long timeout_ns) {
  if (threadIdx.x == 0) {
    signal_counter(counter);
    wait_counter(counter, (uint32_t)expected, timeout_ns, err);
    const uint32_t old = atomicAdd(counter + 1, 1u);
    if (old == gridDim.x - 1) {
      counter[0] = 0;
      counter[1] = 0;
      __threadfence();
    }
  }
}

cudaError_t launch_wait_test(uint32_t* counter, uint32_t* err, int n_blocks, int expected,
                             unsigned long long timeout_ns, cudaStream_t st) {
  wait_test_kernel<<<n_blocks, 32, 0, st>>>(counter, err, expected, timeout_ns);
  return cudaGetLastError();
}

}  // namespace fmoe
