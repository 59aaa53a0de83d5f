// Single-launch persistent kernel for batch-1 MoE blocks and stacks of them.
//
// flash-moe (discuss.pytorch.kr write-up, "per-layer pipeline" and "deferred
// CMD3") runs routing, the expert forward and the combine + residual + norm
// per layer as GPU command buffers submitted without waiting; the slotstream
// write-up (simpler24.com, "the disk was not the slow part") measured batch-1
// quantised matmuls at 20 % of memory bandwidth because of dispatch cost.
// Here one cooperative launch (one block per SM) runs every layer.
//
// Ownership.  The K+S selected experts ("slots"; slot 0 is the shared expert
// when there is one) have NS*I intermediate columns in all.  Block c of n
// owns the contiguous range [NS*I*c/n, NS*I*(c+1)/n) of them in slot-major
// order: for each owned column i of a slot it computes the gate and up row
// dot products, h[i] = w_slot * silu(gate . x) * (up . x), and the column's
// contribution Wd[:, i] * h[i] to all H outputs.  h never leaves the block;
// the down projection is stored by column so that a block's columns are one
// contiguous byte range.  Every byte of the selected experts is read by one
// block (the down (scale,bias) words of a 64-column group by each block that
// owns a column of it).
//
// One exchange per layer.  Each block adds its H partial outputs into an
// accumulator with 64-bit integer atomics in fixed point (value << 8 | count
// of contributions, see fmoe_internal.cuh): the sum does not depend on the
// order of arrival, and a word is complete when its count equals the number
// of blocks, so readers need no counter or flag.  Every block then reads the
// whole sum as the next layer's input (residual + sum, RMS-normalised for a
// stack).  Three accumulators rotate: layer l adds into A[l%3] while each
// block clears its own slice of A[(l+1)%3]; A[(l+1)%3] was last read at the
// start of layer l-1, which every block finished before its layer-l-1 sums
// (and so before the clear) could be complete.
//
// Warp roles:
//   12 gate/up warps   dequantised gate/up dot products of the ring's stages
//                      against the layer input (pre-scaled, in registers);
//                      partial sums per row into shared memory
//   8 down warps       each thread owns H/256 output rows; for every owned
//                      column, in order, folds its codes times h into
//                      per-row sums, applies the group's scale and bias per
//                      64-column group, and at the end of the layer adds the
//                      rows into the accumulator
//   producer           one warp; its lanes take turns issuing the bulk
//                      asynchronous copies (TMA engine, mbarrier completion):
//                      gate/up records through a ring of stages, the block's
//                      down columns and their (scale,bias) words into the
//                      down area.  The shared expert needs no routing, so a
//                      block that owns shared columns requests them for the
//                      next layer as soon as ring stages are free.
//   finaliser          routes (top-K of the next layer at the end of the
//                      current one, published once the layer input is
//                      complete), clears the block's accumulator slice,
//                      turns each stage's partial sums into h
// The first 20 warps also gather each layer's input from the accumulator.
//
// No layer's routed experts are requested before its input is complete.
// Every wait is bounded (%globaltimer); a wait that runs out records the
// time-out in the workspace error word, and every later wait of the block
// returns at once, so the launch always ends.  Block-wide barriers appear
// only at the top level (after set-up, before exit), reached once by every
// thread; everything else synchronises through mbarriers or release/acquire
// counters.
#include <mutex>

#include "fmoe_async.cuh"
#include "fmoe_kernels.cuh"

namespace fmoe {

namespace {

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

// Acquire loads of accumulator words: a reader that sees every block's
// contribution also sees what those blocks wrote before adding (their clears
// of other accumulators), without a fence that would wait for this thread's
// unrelated copies in flight.
__device__ __forceinline__ void ld_acquire_v2(const unsigned long long* p, unsigned long long& a,
                                              unsigned long long& b) {
  asm volatile("ld.acquire.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
}

__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

__device__ __forceinline__ uint32_t ld_acquire_shared(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.cta.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(smem_u32(p)) : "memory");
  return v;
}

__device__ __forceinline__ void st_release_shared(uint32_t* p, uint32_t v) {
  asm volatile("st.release.cta.shared::cta.u32 [%0], %1;" ::"r"(smem_u32(p)), "r"(v) : "memory");
}

// Eight consecutive accumulator words (16-byte aligned) once every count is
// `need`; their sums in s.  One thread, bounded.  Returns false if the block
// gave up.
__device__ __forceinline__ bool poll8(const unsigned long long* p, int need, float (&s)[8],
                                      unsigned long long timeout_ns, uint32_t* err, volatile int* abort) {
  uint64_t t0 = 0;
  bool started = false;
  while (true) {
    unsigned long long w[8];
#pragma unroll
    for (int i = 0; i < 8; i += 2) ld_acquire_v2(p + i, w[i], w[i + 1]);
    bool ok = true;
#pragma unroll
    for (int i = 0; i < 8; ++i) ok = ok && fix_count(w[i]) == need;
    if (ok) {
#pragma unroll
      for (int i = 0; i < 8; ++i) s[i] = fix_value(w[i]);
      return true;
    }
    if (*abort) return false;
    const uint64_t t = global_timer_ns();
    if (!started) {
      t0 = t;
      started = true;
    } else if (t - t0 > timeout_ns) {
      atomicOr(err, kErrWaitTimeout);
      *abort = 1;
      return false;
    }
    __nanosleep(kPollNs);
  }
}

// Wait (bounded) until a release counter in shared memory reaches `target`,
// pausing kWaitNs between checks so that the waiting warps leave the issue
// slots to the warps doing the arithmetic.
__device__ __forceinline__ bool wait_count(const uint32_t* ctr, uint32_t target, unsigned long long timeout_ns,
                                           uint32_t* err, volatile int* abort) {
  if (ld_acquire_shared(ctr) >= target) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (kWaitNs) __nanosleep(kWaitNs);
    if (ld_acquire_shared(ctr) >= target) return true;
    if ((it & 255u) == 0u) {
      if (*abort) return false;
      if (global_timer_ns() - t0 > timeout_ns) {
        atomicOr(err, kErrWaitTimeout);
        *abort = 1;
        return false;
      }
    }
  }
}

// Positions of the 8 elements e..e+7 (e a multiple of 8) in the slice-major
// input layout: float4 j of slice s at j*tl + s.
__device__ __forceinline__ int xs_pos4(int e, int tl) { return ((e & 31) >> 2) * tl + (e >> 5); }

}  // namespace

// Down-projection step of one column for one 32-bit word of codes (rows
// 32/BITS of them): acc[r] += code[r] * h, the codes masked in place and h
// pre-scaled per position (hv: BITS == 4: 4 values, 2: 8 values).
template <int BITS>
__device__ __forceinline__ void down_word(uint32_t w, const float2* hv, float2* acc) {
  const uint32_t hi = w >> 16;
  if constexpr (BITS == 4) {
    acc[0] = __ffma2_rn(mk2(w, 0xFu, 0xF0u), hv[0], acc[0]);
    acc[1] = __ffma2_rn(mk2(w, 0xF00u, 0xF000u), hv[1], acc[1]);
    acc[2] = __ffma2_rn(mk2(hi, 0xFu, 0xF0u), hv[0], acc[2]);
    acc[3] = __ffma2_rn(mk2(hi, 0xF00u, 0xF000u), hv[1], acc[3]);
  } else {
    acc[0] = __ffma2_rn(mk2(w, 0x3u, 0xCu), hv[0], acc[0]);
    acc[1] = __ffma2_rn(mk2(w, 0x30u, 0xC0u), hv[1], acc[1]);
    acc[2] = __ffma2_rn(mk2(w, 0x300u, 0xC00u), hv[2], acc[2]);
    acc[3] = __ffma2_rn(mk2(w, 0x3000u, 0xC000u), hv[3], acc[3]);
    acc[4] = __ffma2_rn(mk2(hi, 0x3u, 0xCu), hv[0], acc[4]);
    acc[5] = __ffma2_rn(mk2(hi, 0x30u, 0xC0u), hv[1], acc[5]);
    acc[6] = __ffma2_rn(mk2(hi, 0x300u, 0xC00u), hv[2], acc[6]);
    acc[7] = __ffma2_rn(mk2(hi, 0x3000u, 0xC000u), hv[3], acc[7]);
  }
}

// MW: code words of a down column per down thread, ceil(H / (32/BITS) / 256)
// rounded up to 1, 2 or 4.
template <int BITS, int MW>
__global__ void __launch_bounds__(kFusedThreads, 1) fused_moe_kernel(const __grid_constant__ FusedParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int RW = 32 / BITS;                 // rows per code word of a down column
  constexpr int NV = BITS == 4 ? 4 : 8;         // pre-scaled copies of h per column
  const FusedPlan& pl = p.plan;
  const BlobLayout& lay = p.lay;
  // control area
  uint64_t* bar_full = reinterpret_cast<uint64_t*>(smem);   // ring stage filled (count 1 + bytes)
  uint64_t* bar_empty = bar_full + kMaxStages;              // ring stage free (gate/up warps)
  uint64_t* bar_gudone = bar_empty + kMaxStages;            // [2*kMaxStages] stage's partial sums written
  uint64_t* bar_pfree = bar_gudone + 2 * kMaxStages;        // [2*kMaxStages] partial sums read (finaliser)
  uint64_t* bar_x = bar_pfree + 2 * kMaxStages;             // layer input gathered (input warps)
  uint64_t* bar_routed = bar_x + 1;                         // layer's routing published (finaliser)
  uint64_t* bar_zero = bar_routed + 1;                      // next accumulator slice cleared (finaliser)
  uint64_t* bar_dfull = bar_zero + 1;                       // down area filled (count 1 + bytes)
  uint64_t* bar_ddone = bar_dfull + 1;                      // down area free again (down warps)
  Piece* s_pc = reinterpret_cast<Piece*>(smem + 1024);      // [kMaxPieces]
  int* s_np = reinterpret_cast<int*>(smem + 1152);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + 1156);
  uint32_t* s_hdone = reinterpret_cast<uint32_t*>(smem + 1160);  // stages whose h is written (cumulative)
  int* s_ids = reinterpret_cast<int*>(smem + 1280);         // [2][kMaxSlots] by layer parity
  float* s_w = reinterpret_cast<float*>(smem + 1536);       // [2][kMaxSlots] routing weights, shared gate
  float* s_red = reinterpret_cast<float*>(smem + 1792);     // [kPollWarps][2]
  float4* s_x4 = reinterpret_cast<float4*>(smem + pl.xs_off);   // layer input h (not normalised), slice-major
  float* s_part = reinterpret_cast<float*>(smem + pl.part_off); // [2*nstage][R][nparts][2]
  float* s_hb = reinterpret_cast<float*>(smem + pl.hbuf_off);   // [len][hb]: NV pre-scaled h, then h
  float* s_dscr = reinterpret_cast<float*>(smem + pl.dscr_off);  // [kDnThreads][RW*MW] transpose scratch
  uint8_t* darea = smem + pl.darea_off;                          // the block's down columns and scale/bias
  uint8_t* ring = smem + pl.ring_off;

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int c = blockIdx.x, n = gridDim.x;
  const int NS = p.K + p.S;
  const int H = p.H, I = p.I;
  const int tl = H / kSlice;
  const int R = pl.R, nparts = pl.nparts, hb = pl.hb;
  const int gw = tl < 32 ? tl : 32;                          // reduction width of a gate/up row
  long long bv0, bv1;
  block_bounds(NS, I, p.S, c, n, bv0, bv1);
  const int len = (int)(bv1 - bv0);                         // columns of this block
  const int nstg = (len + R - 1) / R;
  const int ja = (int)((long long)H * c / n);               // accumulator slice this block clears
  const int nd = (int)((long long)H * (c + 1) / n) - ja;
  const unsigned long long tmo = p.timeout_ns;

  if (tid == 0) {
    for (int i = 0; i < kMaxStages; ++i) {
      mbar_init(&bar_full[i], 1);
      mbar_init(&bar_empty[i], kGuWarps);
    }
    for (int i = 0; i < 2 * kMaxStages; ++i) {
      mbar_init(&bar_gudone[i], kGuWarps);
      mbar_init(&bar_pfree[i], 1);
    }
    mbar_init(bar_x, kPollWarps);
    mbar_init(bar_routed, 1);
    mbar_init(bar_zero, 1);
    mbar_init(bar_dfull, 1);
    mbar_init(bar_ddone, kDnWarps);
    int dbytes = 0;
    *s_np = block_pieces(NS, I, p.S, c, n, lay, s_pc, kMaxPieces, dbytes);
    *s_abort = 0;
    *s_hdone = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  const int np = *s_np;
  const uint32_t lb = *reinterpret_cast<volatile uint32_t*>(p.lbase);

  uint32_t g_issue = 0;   // ring stages issued (producer)
  uint32_t n_copies = 0;  // bulk copies issued (producer): picks the issuing lane
  uint32_t g_cons = 0;    // ring stages consumed (gate/up warps, finaliser)
  int nx_id = -1;         // finaliser: top-K pick of its lane for the coming layer
  float nx_l = 0.f;
  auto slot_h = [&](int slot) -> int { return p.S ? (slot == 0 ? p.K : slot - 1) : slot; };
  for (int l = 0; l < p.L; ++l) {
    const FusedLayerPtrs lp = p.layer[l];
    const uint32_t lpar = (uint32_t)(l & 1);
    unsigned long long* acc_cur = p.acc + (size_t)((lb + l) % 3) * H;
    const unsigned long long* acc_prev = p.acc + (size_t)((lb + l + 2) % 3) * H;
    unsigned long long* acc_next = p.acc + (size_t)((lb + l + 1) % 3) * H;

    if (warp < kPollWarps) {
      // ------------------------------------------------------------------
      // layer input: x (block), h (first layer of a stack) or the previous
      // layer's complete sum added to its input; staged slice-major, with
      // the sums of squares and of products with the shared-gate vector
      // ------------------------------------------------------------------
      float ss = 0.f, wg = 0.f;
      if (l > 0 && warp * 256 < H) {
        // one lane waits for the warp's first words before every lane polls
        // its own: the accumulators are not read over and over while the
        // blocks' additions are still landing
        if (lane == 0) {
          float sm[8];
          poll8(acc_prev + warp * 256, n, sm, tmo, p.err, s_abort);
        }
        __syncwarp();
      }
      for (int e = tid * 8; e < H; e += kPollWarps * 32 * 8) {
        const int q0 = xs_pos4(e, tl), q1 = xs_pos4(e + 4, tl);
        float4 v0, v1;
        if (l == 0) {
          const float4* src = reinterpret_cast<const float4*>((p.norm ? p.out : p.x) + e);
          v0 = __ldcg(src);
          v1 = __ldcg(src + 1);
        } else {
          float sm[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
          poll8(acc_prev + e, n, sm, tmo, p.err, s_abort);
          v0 = s_x4[q0];
          v1 = s_x4[q1];
          v0.x += sm[0]; v0.y += sm[1]; v0.z += sm[2]; v0.w += sm[3];
          v1.x += sm[4]; v1.y += sm[5]; v1.z += sm[6]; v1.w += sm[7];
        }
        s_x4[q0] = v0;
        s_x4[q1] = v1;
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
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_x);

      if (warp < kGuWarps) {
        // ---------------- gate/up: stream the ring, partial sums to smem ----
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
        mbar_wait(bar_x, lpar, tmo, p.err, s_abort);
        float tot = 0.f;
#pragma unroll 4
        for (int q = 0; q < kPollWarps; ++q) tot += s_red[2 * q];
        const float rinv = p.norm ? 1.0f / sqrtf(tot / (float)H + p.eps) : 1.0f;
        SliceX xs;
        float xsum = 0.f;
#pragma unroll
        for (int j = 0; j < kSlice / 4; ++j) {
          const float4 v = s_x4[j * tl + sl];
          xsum += put_x4<BITS>(xs, j, make_float4(v.x * rinv, v.y * rinv, v.z * rinv, v.w * rinv));
        }
        for (int k = 0; k < nstg; ++k) {
          const uint32_t st = g_cons % pl.nstage;
          mbar_wait(&bar_full[st], (g_cons / pl.nstage) & 1u, tmo, p.err, s_abort);
          ++g_cons;
          const uint8_t* buf = ring + (size_t)st * pl.stage_bytes;
          const int u0 = k * R + rs0, u1 = k * R + rs1;
          float ga0 = 0.f, ua0 = 0.f, ga1 = 0.f, ua1 = 0.f;
          if (rs0 < R / 2 && u0 < len) {
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
          if (rs0 < R / 2 && u1 < len) {
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
          // the ring stage is free once every gate/up warp has read it
          __syncwarp();
          if (lane == 0) mbar_arrive(&bar_empty[st]);
          const float v = quad_reduce(ga0, ua0, ga1, ua1, gw, lane);
          const int pos = lane & (gw - 1), qw = gw >> 2;
          const int rsel = pos < 2 * qw ? rs0 : rs1;
          // partial sums: 2*nstage slots, each reused once the finaliser has read it
          const uint32_t g = g_cons - 1, ps = g % (2u * pl.nstage);
          if (g >= 2u * pl.nstage) mbar_wait(&bar_pfree[ps], ((g / (2u * pl.nstage)) - 1u) & 1u, tmo, p.err, s_abort);
          if (rs0 < R / 2 && k * R + rsel < len && (pos & (qw - 1)) == 0)
            s_part[(((size_t)ps * R + rsel) * nparts + pi) * 2 + ((pos / qw) & 1)] = v;
          __syncwarp();
          if (lane == 0) mbar_arrive(&bar_gudone[ps]);
        }
      } else {
        // ---------------- down: owned columns, in order, into per-row sums ----
        // Thread dt owns code words [MW*dt, MW*dt + MW) of every column, i.e.
        // RW*MW consecutive output rows; the block's columns and their groups'
        // scale/bias words sit in the down area (bulk copies by the producer).
        const int dt = tid - kGuWarps * 32;
        const int W = H / RW;                                  // code words per column
        const int wb = MW * dt;                                // this thread's first code word
        const bool dact = wb < W;
        float outp[MW * RW];
#pragma unroll
        for (int r = 0; r < MW * RW; ++r) outp[r] = 0.f;
        // this block's clear of the next accumulator is ordered before this
        // thread's additions (the fence waits here, off the critical path)
        mbar_wait(bar_zero, lpar, tmo, p.err, s_abort);
        fence_acq_rel_gpu();
        // where each piece's expert blob is (the layer's routing was published
        // before its input was complete, hence before bar_zero)
        const int* ids_d = s_ids + (size_t)(l & 1) * kMaxSlots;
        auto piece_blob = [&](int slot) -> const uint8_t* {
          if (p.S && slot == 0) return lp.shared;
          return lp.experts + (size_t)ids_d[slot] * p.blob;
        };
        if (kFusedSbGlobal && dact) {
          for (int pidx = 0; pidx < np; ++pidx) {
            const Piece pc = s_pc[pidx];
            const uint8_t* sb0 = piece_blob(pc.slot) + lay.dsb_off + (size_t)pc.g0 * lay.dsb_group + (size_t)wb * RW * 4;
            for (int gi = 0; gi < pc.ng; ++gi)
              asm volatile("prefetch.global.L2 [%0];" ::"l"(sb0 + (size_t)gi * lay.dsb_group));
          }
        }
        mbar_wait(bar_dfull, lpar, tmo, p.err, s_abort);
        const uint32_t hd_base = (uint32_t)l * (uint32_t)nstg;
        int seen = 0;                                          // stages of this layer known finalised
        for (int pidx = 0; pidx < np; ++pidx) {
          const Piece pc = s_pc[pidx];
          const uint8_t* cbase = darea + pc.col_off;
          for (int gi = 0; gi < pc.ng; ++gi) {
            const int g = pc.g0 + gi;
            const int ia = max(pc.i0, g * kGroup), ib = min(pc.i0 + pc.cnt, g * kGroup + kGroup);
            float2 acc[MW][RW / 2];
#pragma unroll
            for (int j = 0; j < MW; ++j)
#pragma unroll
              for (int t = 0; t < RW / 2; ++t) acc[j][t] = make_float2(0.f, 0.f);
            float hs = 0.f;
            for (int i = ia; i < ib; ++i) {
              const int u = pc.loc + (i - pc.i0);
              while (seen * R <= u) {
                wait_count(s_hdone, hd_base + (uint32_t)seen + 1u, tmo, p.err, s_abort);
                ++seen;
              }
              const float4* hp4 = reinterpret_cast<const float4*>(s_hb + (size_t)u * hb);
              float2 hv[NV / 2];
              {
                const float4 a = hp4[0];
                hv[0] = make_float2(a.x, a.y);
                hv[1] = make_float2(a.z, a.w);
                if constexpr (BITS == 2) {
                  const float4 b = hp4[1];
                  hv[2] = make_float2(b.x, b.y);
                  hv[3] = make_float2(b.z, b.w);
                }
              }
              hs += s_hb[(size_t)u * hb + NV];
              if (dact) {
                const uint32_t* col = reinterpret_cast<const uint32_t*>(cbase + (size_t)(i - pc.i0) * lay.dcol) + wb;
                uint32_t w[MW];
                if constexpr (MW == 4) {
                  const uint4 v = *reinterpret_cast<const uint4*>(col);
                  w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
                } else if constexpr (MW == 2) {
                  const uint2 v = *reinterpret_cast<const uint2*>(col);
                  w[0] = v.x; w[1] = v.y;
                } else {
                  w[0] = col[0];
                }
#pragma unroll
                for (int j = 0; j < MW; ++j) down_word<BITS>(w[j], hv, acc[j]);
              }
            }
            // the group's scale and bias per row: out += s * 2^64 * acc + b * sum(h)
            if (dact) {
              const uint4* sbw = reinterpret_cast<const uint4*>(
                  (kFusedSbGlobal ? piece_blob(pc.slot) + lay.dsb_off + (size_t)pc.g0 * lay.dsb_group
                                  : darea + pc.sb_off) +
                  (size_t)gi * lay.dsb_group + (size_t)wb * RW * 4);
#pragma unroll
              for (int j = 0; j < MW; ++j) {
#pragma unroll
                for (int t4 = 0; t4 < RW / 4; ++t4) {
                  const uint4 s4 = sbw[j * (RW / 4) + t4];
                  const float2 a01 = acc[j][2 * t4], a23 = acc[j][2 * t4 + 1];
                  float* o = outp + j * RW + 4 * t4;
                  o[0] += fmaf(bf16lo(s4.x) * 18446744073709551616.0f, a01.x, bf16hi(s4.x) * hs);
                  o[1] += fmaf(bf16lo(s4.y) * 18446744073709551616.0f, a01.y, bf16hi(s4.y) * hs);
                  o[2] += fmaf(bf16lo(s4.z) * 18446744073709551616.0f, a23.x, bf16hi(s4.z) * hs);
                  o[3] += fmaf(bf16lo(s4.w) * 18446744073709551616.0f, a23.y, bf16hi(s4.w) * hs);
                }
              }
            }
          }
        }
        // the down area may be refilled for the next layer
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_ddone);
        // Each warp owns 32*E consecutive rows (E = RW*MW per thread); a
        // transpose through the warp's own 128-float scratch, four rows per
        // lane at a time, lets every red instruction of the warp add 32
        // consecutive rows (coalesced), with no wait on the other down warps.
        {
          constexpr int E = RW * MW;
          float* scr = s_dscr + (size_t)(warp - kGuWarps) * 128;
          const int r0 = (warp - kGuWarps) * 32 * E;          // the warp's first row
#pragma unroll
          for (int t0 = 0; t0 < E; t0 += 4) {
            // rows r0 + 32*t0 .. r0 + 32*(t0+4) - 1 are held by lanes
            // 32*t0/E .. 32*(t0+4)/E - 1
            const int l0 = 32 * t0 / E, l1 = 32 * (t0 + 4) / E;
            __syncwarp();
            if (lane >= l0 && lane < l1) {
#pragma unroll
              for (int e = 0; e < E; e += 4)
                *reinterpret_cast<float4*>(scr + (lane - l0) * E + e) =
                    make_float4(outp[e], outp[e + 1], outp[e + 2], outp[e + 3]);
            }
            __syncwarp();
            if (!*s_abort && r0 < H) {
#pragma unroll
              for (int t = 0; t < 4; ++t) {
                const int row = r0 + 32 * (t0 + t) + lane;
                if (row < H) red_add_u64(acc_cur + row, fix_word(scr[32 * t + lane], p.err));
              }
            }
          }
          __syncwarp();
        }
      }
    } else if (warp == kProducerWarp) {
      // ------------------------------------------------------------------
      // producer: the layer's copies in consumption order; lane 0 declares
      // each barrier's bytes, successive copies are issued by successive
      // lanes (the copies one thread issues are carried out one after
      // another, those of different threads side by side)
      // ------------------------------------------------------------------
      auto aborted = [&]() -> bool { return __shfl_sync(0xFFFFFFFFu, *s_abort, 0) != 0; };
      bool routed = false;       // routed ids are published all at once
      auto ensure_routed = [&](int slot) {
        if (slot >= p.S && !routed) {
          // the ids are known early; the copies wait for the layer's input
          mbar_wait(bar_routed, lpar, tmo, p.err, s_abort);
          mbar_wait(bar_x, lpar, tmo, p.err, s_abort);
          routed = true;
        }
      };
      const int* ids_l = s_ids + (size_t)(l & 1) * kMaxSlots;
      auto slot_blob = [&](int slot) -> const uint8_t* {
        if (p.S && slot == 0) return lp.shared;
        return lp.experts + (size_t)ids_l[slot] * p.blob;
      };
      auto copy = [&](uint8_t* dst, const uint8_t* src, uint32_t bytes, uint64_t* bar) {
        for (uint32_t off = 0; off < bytes; off += kFusedCopyBytes) {
          const uint32_t b = bytes - off < kFusedCopyBytes ? bytes - off : kFusedCopyBytes;
          if (lane == (int)(n_copies % kFusedIssueLanes)) bulk_g2s(dst + off, src + off, b, bar);
          ++n_copies;
        }
      };
      auto issue_darea = [&]() {
        // the previous layer's down work is done with the area
        if (l > 0) mbar_wait(bar_ddone, (uint32_t)((l - 1) & 1), tmo, p.err, s_abort);
        uint32_t total = 0;
        for (int q = 0; q < np; ++q)
          total += (uint32_t)(s_pc[q].cnt * lay.dcol + (kFusedSbGlobal ? 0 : s_pc[q].ng * lay.dsb_group));
        if (aborted()) {
          if (lane == 0) mbar_arrive_expect_tx(bar_dfull, 0);
          return;
        }
        if (lane == 0) mbar_arrive_expect_tx(bar_dfull, total);
        __syncwarp();
        for (int q = 0; q < np; ++q) {
          const Piece pc = s_pc[q];
          ensure_routed(pc.slot);
          if (aborted()) continue;
          const uint8_t* b = slot_blob(pc.slot);
          copy(darea + pc.col_off, b + lay.dq_off + (size_t)pc.i0 * lay.dcol, (uint32_t)(pc.cnt * lay.dcol),
               bar_dfull);
          if (!kFusedSbGlobal)
            copy(darea + pc.sb_off, b + lay.dsb_off + (size_t)pc.g0 * lay.dsb_group,
                 (uint32_t)(pc.ng * lay.dsb_group), bar_dfull);
        }
      };
      bool darea_issued = false;
      for (int k = 0; k < nstg; ++k) {
        const uint32_t st = g_issue % pl.nstage;
        const uint32_t use = g_issue / pl.nstage;
        ++g_issue;
        if (use >= 1) mbar_wait(&bar_empty[st], (use - 1) & 1u, tmo, p.err, s_abort);
        const int a0 = k * R, a1 = min(len, a0 + R);
        if (aborted()) {
          if (lane == 0) mbar_arrive_expect_tx(&bar_full[st], 0);
        } else {
          if (lane == 0) mbar_arrive_expect_tx(&bar_full[st], (uint32_t)((a1 - a0) * lay.gu_row));
          __syncwarp();
          uint8_t* buf = ring + (size_t)st * pl.stage_bytes;
          for (int q = 0; q < np; ++q) {
            const Piece pc = s_pc[q];
            const int b0 = max(a0, pc.loc), b1 = min(a1, pc.loc + pc.cnt);
            if (b0 >= b1) continue;
            ensure_routed(pc.slot);
            if (aborted()) continue;
            copy(buf + (size_t)(b0 - a0) * lay.gu_row, slot_blob(pc.slot) + (size_t)(pc.i0 + b0 - pc.loc) * lay.gu_row,
                 (uint32_t)((b1 - b0) * lay.gu_row), &bar_full[st]);
          }
        }
        if (!darea_issued && (k + 1 >= kFusedDareaAfter || k + 1 >= pl.nstage)) {
          issue_darea();
          darea_issued = true;
        }
      }
      if (!darea_issued) issue_darea();
      __syncwarp();
    } else {
      // ------------------------------------------------------------------
      // finaliser: routing, the accumulator clear, h of each stage
      // ------------------------------------------------------------------
      // the routing of a layer is published as soon as it is known (at the
      // end of the previous layer): the producer still waits for the
      // layer's input before it requests a routed expert
      auto publish = [&](int ll) {
        warp_topk(p.logits + (size_t)ll * p.E, p.E, p.K, nx_id, nx_l);
        const float my_w = warp_topk_softmax(nx_l, p.K);
        if (lane < p.K) {
          s_ids[(ll & 1) * kMaxSlots + p.S + lane] = nx_id;
          s_w[(ll & 1) * kMaxSlots + p.S + lane] = my_w;
          if (c == 0 && p.ids_out != nullptr) {
            p.ids_out[(size_t)ll * p.K + lane] = nx_id;
            p.w_out[(size_t)ll * p.K + lane] = my_w;
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_routed);
      };
      if (l == 0) publish(0);
      float* w_l = s_w + (size_t)(l & 1) * kMaxSlots;
      mbar_wait(bar_x, lpar, tmo, p.err, s_abort);
      float tot = 0.f, wgt = 0.f;
#pragma unroll 4
      for (int q = 0; q < kPollWarps; ++q) {
        tot += s_red[2 * q];
        wgt += s_red[2 * q + 1];
      }
      const float rinv = p.norm ? 1.0f / sqrtf(tot / (float)H + p.eps) : 1.0f;
      const float gate = p.S ? sigmoid_f(wgt * rinv) : 0.f;
      if (lane == 0) {
        if (p.S) w_l[0] = gate;
        if (c == 0 && p.gate_out != nullptr) p.gate_out[l] = gate;
      }
      __syncwarp();
      // clear this block's slice of the next layer's accumulator (its last
      // readers finished before this layer's input was complete)
      for (int r = lane; r < nd; r += 32) acc_next[ja + r] = 0ull;
      __threadfence();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_zero);
      const bool last = (l == p.L - 1) && p.hmid != nullptr;
      for (int k = 0; k < nstg; ++k) {
        const uint32_t ps = g_cons % (2u * pl.nstage);
        if (kFinalSpin)
          mbar_wait_spin(&bar_gudone[ps], (g_cons / (2u * pl.nstage)) & 1u, tmo, p.err, s_abort);
        else
          mbar_wait(&bar_gudone[ps], (g_cons / (2u * pl.nstage)) & 1u, tmo, p.err, s_abort);
        ++g_cons;
        const int nrec = min(R, len - k * R);
        for (int r = lane; r < nrec; r += 32) {
          const int u = k * R + r;
          int q = 0;
          while (q + 1 < np && u >= s_pc[q + 1].loc) ++q;
          const int slot = s_pc[q].slot, i = s_pc[q].i0 + (u - s_pc[q].loc);
          const float* part = s_part + ((size_t)ps * R + r) * nparts * 2;
          float a = 0.f, uu = 0.f;
          for (int t = 0; t < nparts; ++t) {
            a += part[2 * t];
            uu += part[2 * t + 1];
          }
          const float hv = silu_f(a) * uu;
          const float hw = w_l[slot] * hv;
          float* dst = s_hb + (size_t)u * hb;
#pragma unroll
          for (int t = 0; t < NV; ++t) dst[t] = hw * pos_scale<BITS>(t);
          dst[NV] = hw;
          if (last) p.hmid[(size_t)slot_h(slot) * I + i] = hv;
        }
        __threadfence_block();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&bar_pfree[ps]);
          st_release_shared(s_hdone, (uint32_t)l * (uint32_t)nstg + (uint32_t)k + 1u);
        }
      }
      // the next layer's routing, off its critical path
      if (l + 1 < p.L) publish(l + 1);
    }
  }

  // ---- the last layer's output: this block's chunks of 8 outputs ----
  if (warp < kPollWarps) {
    const unsigned long long* acc_last = p.acc + (size_t)((lb + p.L - 1) % 3) * H;
    for (int q = c + n * tid; q < H / 8; q += n * kPollWarps * 32) {
      const int e = q * 8;
      float sm[8];
      if (!poll8(acc_last + e, n, sm, tmo, p.err, s_abort)) break;
      float4 b0, b1;
      if (p.norm) {
        b0 = s_x4[xs_pos4(e, tl)];
        b1 = s_x4[xs_pos4(e + 4, tl)];
      } else {
        b0 = __ldg(reinterpret_cast<const float4*>(p.residual + e));
        b1 = __ldg(reinterpret_cast<const float4*>(p.residual + e) + 1);
      }
      float4* o = reinterpret_cast<float4*>(p.out + e);
      o[0] = make_float4(b0.x + sm[0], b0.y + sm[1], b0.z + sm[2], b0.w + sm[3]);
      o[1] = make_float4(b1.x + sm[4], b1.y + sm[5], b1.z + sm[6], b1.w + sm[7]);
    }
  }

  // No copy may still be writing this block's shared memory when it exits:
  // wait (bounded, whether or not the block gave up) for the last phase of
  // every stage and of the down area.
  if (warp == kProducerWarp && lane == 0) {
    volatile int no_abort = 0;
    const uint32_t used = g_issue < (uint32_t)pl.nstage ? g_issue : (uint32_t)pl.nstage;
    for (uint32_t st = 0; st < used; ++st) {
      const uint32_t lastu = g_issue - 1 - ((g_issue - 1 - st) % pl.nstage);   // last issue index of stage st
      mbar_wait(&bar_full[st], (lastu / pl.nstage) & 1u, tmo, p.err, &no_abort);
    }
    mbar_wait(bar_dfull, (uint32_t)((p.L - 1) & 1), tmo, p.err, &no_abort);
  }

  // the last block out advances the layer count and resets the exit count
  __syncwarp();
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    const uint32_t old = atomicAdd(p.exit_ctr, 1u);
    if (old == (uint32_t)n - 1) {
      *p.exit_ctr = 0;
      *p.lbase = (lb + (uint32_t)p.L) % 3u;
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
  if (bits != 4 && bits != 2) return pl;
  const int tl = H / kSlice;
  if (H % 64 || I % 64 || !pow2(tl) || tl < 4) return pl;
  if (K < 1 || K + S > kMaxSlots || sms < 1 || sms > kFixMaxContrib) return pl;
  const int NS = K + S;
  const int grid = sms;
  const BlobLayout lay = blob_layout(bits, H, I);
  // a down thread holds at most 4 (4-bit) or 2 (2-bit) code words of a column
  if (H / (32 / bits) > kDnThreads * (bits == 4 ? 4 : 2)) return pl;
  const int nparts = tl >= 32 ? tl / 32 : 1;
  if (nparts > kGuWarps) return pl;
  const int R = 2 * (tl >= 32 ? kGuWarps / nparts : kGuWarps * (32 / tl));
  pl.R = R;
  pl.nparts = nparts;
  pl.stage_bytes = round_up_i((long long)R * lay.gu_row, 128);
  pl.len_max = 0;
  int darea = 0;
  for (int c = 0; c < grid; ++c) {
    Piece pc[kMaxPieces];
    int b = 0;
    if (block_pieces(NS, I, S, c, grid, lay, pc, kMaxPieces, b) > kMaxPieces) return pl;
    darea = b > darea ? b : darea;
    long long v0, v1;
    block_bounds(NS, I, S, c, grid, v0, v1);
    pl.len_max = (int)(v1 - v0) > pl.len_max ? (int)(v1 - v0) : pl.len_max;
  }
  pl.darea_bytes = round_up_i(darea > 128 ? darea : 128, 128);
  pl.hb = bits == 4 ? 8 : 12;
  pl.xs_off = kCtrlBytes;
  pl.part_off = round_up_i(pl.xs_off + (long long)H * 4, 128);
  for (int ns = kFusedStageCap; ns >= 2; --ns) {
    pl.hbuf_off = round_up_i(pl.part_off + (long long)2 * ns * R * nparts * 2 * 4, 128);
    pl.dscr_off = round_up_i(pl.hbuf_off + (long long)(pl.len_max + 1) * pl.hb * 4, 128);
    pl.darea_off = round_up_i(pl.dscr_off + (long long)kDnWarps * 128 * 4, 128);
    pl.ring_off = pl.darea_off + pl.darea_bytes;
    const long long need = (long long)pl.ring_off + (long long)ns * pl.stage_bytes;
    if (need <= smem_max) {
      pl.nstage = ns;
      pl.smem = (size_t)need;
      pl.grid = grid;
      pl.ok = true;
      return pl;
    }
  }
  return pl;
}

template <int BITS, int MW>
static cudaError_t launch_fused_t(FusedParams& p, const FusedPlan& pl, cudaStream_t st) {
  // the shared-memory limit and the residency check, once per device and size
  // (function attributes belong to the device's context)
  static std::mutex mu;
  static int configured_smem[64];
  static size_t checked_smem[64];
  auto kern = fused_moe_kernel<BITS, MW>;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (configured_smem[dev] < (int)pl.smem) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pl.smem);
      if (e != cudaSuccess) return e;
      configured_smem[dev] = (int)pl.smem;
    }
    if (checked_smem[dev] != pl.smem) {
      int per_sm = 0;
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kFusedThreads, pl.smem);
      if (e != cudaSuccess) return e;
      if (per_sm < 1) return cudaErrorCooperativeLaunchTooLarge;
      checked_smem[dev] = pl.smem;
    }
  }
  // cooperative: all blocks resident at once (every block waits for words
  // that the other blocks add)
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
  return cudaLaunchKernelEx(&cfg, kern, p);
}

cudaError_t launch_fused(FusedParams& p, const FusedPlan& pl, cudaStream_t st) {
  p.plan = pl;
  const int words = p.H / (32 / p.bits);                     // code words per down column
  const int mw = (words + kDnThreads - 1) / kDnThreads;
  if (p.bits == 4) {
    if (mw <= 1) return launch_fused_t<4, 1>(p, pl, st);
    if (mw <= 2) return launch_fused_t<4, 2>(p, pl, st);
    return launch_fused_t<4, 4>(p, pl, st);
  }
  if (mw <= 1) return launch_fused_t<2, 1>(p, pl, st);
  return launch_fused_t<2, 2>(p, pl, st);
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
