// Single-launch persistent kernel for batch-1 MoE blocks and stacks of them.
//
// flash-moe (discuss.pytorch.kr write-up, "per-layer pipeline" and "deferred
// CMD3") runs routing, the expert forward and the combine + residual + norm
// per layer as GPU command buffers submitted without waiting; the slotstream
// write-up (simpler24.com) measured batch-1 quantised matmuls at 20 % of
// memory bandwidth because of dispatch cost.  Here one cooperative launch
// (one 512-thread block per SM) runs, for each layer:
//
//   prologue   every block: RMSNorm statistics of the input (stacks), top-K +
//              softmax of the router logits, sigmoid shared-expert gate, and
//              its pre-scaled input slice in registers
//   gate/up    block c owns intermediate rows [I*c/n, I*(c+1)/n) of every
//              selected expert ("slot"); their packed rows stream from HBM into
//              a shared-memory ring with bulk asynchronous copies (TMA engine,
//              mbarrier completion); SwiGLU is applied in the epilogue and h
//              goes to global memory (L2)
//   down       block c owns output rows [H*c/n, H*(c+1)/n); their packed rows
//              of every slot are copied into shared memory while gate/up runs.
//              After a slot's h is complete device-wide (a per-slot counter,
//              bounded wait) the block folds w_slot * (down_row . h_slot) into
//              per-row accumulators, one slot behind the gate/up stream, so
//              only the last slot's down work trails the last weight byte.
//   combine    out[j] = residual[j] + sum over slots, written by the row's owner
//
// Weight bytes of a layer are requested only after the previous layer's
// output is complete (a device-wide counter), as a real decoder would have
// to.  Every wait is bounded (%globaltimer) and records a time-out in the
// workspace error word instead of hanging.
#include "fmoe_kernels.cuh"

namespace fmoe {

namespace {

constexpr int kCtrlBytes = 6144;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait on an mbarrier phase; records a time-out and returns.
__device__ __forceinline__ void mbar_wait(uint64_t* bar, uint32_t parity, uint64_t timeout_ns,
                                          uint32_t* err) {
  if (mbar_try_wait(bar, parity)) return;
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > timeout_ns) {
      atomicOr(err, kErrCopyTimeout);
      return;
    }
  }
}

__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// A byte range rounded out to 16-byte boundaries for the bulk-copy engine.
struct Span {
  const uint8_t* src;   // 16-byte aligned start
  uint32_t off;         // offset of the wanted bytes inside the copy
  uint32_t len;         // multiple of 16
};

__device__ __forceinline__ Span span_of(const uint8_t* p, uint32_t bytes) {
  Span s;
  const uintptr_t a = reinterpret_cast<uintptr_t>(p) & ~(uintptr_t)15;
  s.src = reinterpret_cast<const uint8_t*>(a);
  s.off = (uint32_t)(reinterpret_cast<uintptr_t>(p) - a);
  s.len = (s.off + bytes + 15u) & ~15u;
  return s;
}

// Offset of the wanted bytes inside a rounded copy (consumer side).
__device__ __forceinline__ uint32_t span_off(size_t byte_offset) { return (uint32_t)(byte_offset & 15); }

struct Geo {
  int tl_gu, teams_gu, team, sl, wpt, wit, red_w;   // gate/up teams (one row per team)
  int tl_d, teams_d, dteam, dsl;                     // down teams
  int ra, nr, nch, ja, nd;                           // this block's rows
  size_t qbh, sbbh, qbi, sbbi;                        // row bytes
};

}  // namespace

template <int BITS>
__global__ void __launch_bounds__(kFusedThreads, 1) fused_moe_kernel(const __grid_constant__ FusedParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* mbar_ring = reinterpret_cast<uint64_t*>(smem);
  uint64_t* mbar_d = mbar_ring + kMaxStages;
  int* s_ids = reinterpret_cast<int*>(mbar_d + kMaxSlots);
  float* s_w = reinterpret_cast<float*>(s_ids + kMaxSlots);
  float* s_red = s_w + kMaxSlots;            // 64 floats
  float* s_part = s_red + 64;                // [2][32][2][8] floats
  uint8_t* ring = smem + kCtrlBytes;
  uint8_t* darea = ring + (size_t)p.nstage * p.stage_bytes;

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int c = blockIdx.x, n = gridDim.x;
  const int NS = p.K + p.S;
  const int H = p.H, I = p.I;

  Geo g;
  g.tl_gu = H / kSlice;
  g.teams_gu = kFusedThreads / g.tl_gu;
  g.team = tid / g.tl_gu;
  g.sl = tid % g.tl_gu;
  g.wpt = g.tl_gu >= 32 ? g.tl_gu / 32 : 1;
  g.wit = g.tl_gu >= 32 ? g.sl / 32 : 0;
  g.red_w = g.tl_gu >= 32 ? 32 : g.tl_gu;
  g.tl_d = I / kSlice;
  g.teams_d = kFusedThreads / g.tl_d;
  g.dteam = tid / g.tl_d;
  g.dsl = tid % g.tl_d;
  g.ra = (int)((long long)I * c / n);
  g.nr = (int)((long long)I * (c + 1) / n) - g.ra;
  g.nch = (g.nr + g.teams_gu - 1) / g.teams_gu;
  g.ja = (int)((long long)H * c / n);
  g.nd = (int)((long long)H * (c + 1) / n) - g.ja;
  g.qbh = (size_t)H * BITS / 8;
  g.sbbh = (size_t)H / kGroup * 4;
  g.qbi = (size_t)I * BITS / 8;
  g.sbbi = (size_t)I / kGroup * 4;

  if (tid == 0) {
    for (int i = 0; i < kMaxStages; ++i) mbar_init(&mbar_ring[i], 1);
    for (int i = 0; i < kMaxSlots; ++i) mbar_init(&mbar_d[i], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  // producer state (meaningful in thread 0 only)
  int pr_slot = 0, pr_chunk = 0;
  bool pr_routed = false;
  uint32_t g_issue = 0;
  uint32_t g_cons = 0;          // GU chunks consumed (uniform over the block)

  float accd[kMaxRowsPerTeam];

  for (int l = 0; l < p.L; ++l) {
    const FusedLayerPtrs lp = p.layer[l];
    uint32_t* ctr = p.counters + (size_t)l * (NS + 1);

    auto slot_blob = [&](int ps) -> const uint8_t* {
      if (p.S && ps == 0) return lp.shared;
      return lp.experts + (size_t)s_ids[ps] * p.blob;
    };
    auto hidx = [&](int ps) -> int { return p.S ? (ps == 0 ? p.K : ps - 1) : ps; };

    // ---- producer: issue copies in consumption order, as far as allowed ----
    auto issue_gu = [&](int ps, int pc) {
      const uint8_t* blob = slot_blob(ps);
      const int r0 = g.ra + pc * g.teams_gu;
      const int rn = min(g.teams_gu, g.ra + g.nr - r0);
      const uint32_t st = g_issue % p.nstage;
      uint8_t* buf = ring + (size_t)st * p.stage_bytes;
      const Span a = span_of(blob + p.lay.gate_q + (size_t)r0 * g.qbh, (uint32_t)(rn * g.qbh));
      const Span b = span_of(blob + p.lay.gate_sb + (size_t)r0 * g.sbbh, (uint32_t)(rn * g.sbbh));
      const Span cc = span_of(blob + p.lay.up_q + (size_t)r0 * g.qbh, (uint32_t)(rn * g.qbh));
      const Span d = span_of(blob + p.lay.up_sb + (size_t)r0 * g.sbbh, (uint32_t)(rn * g.sbbh));
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      mbar_arrive_expect_tx(&mbar_ring[st], a.len + b.len + cc.len + d.len);
      bulk_g2s(buf, a.src, a.len, &mbar_ring[st]);
      bulk_g2s(buf + p.gu_cap_q, b.src, b.len, &mbar_ring[st]);
      bulk_g2s(buf + p.gu_cap_q + p.gu_cap_sb, cc.src, cc.len, &mbar_ring[st]);
      bulk_g2s(buf + 2 * p.gu_cap_q + p.gu_cap_sb, d.src, d.len, &mbar_ring[st]);
      ++g_issue;
    };
    auto issue_d = [&](int ps) {
      uint8_t* buf = darea + (size_t)ps * p.dslot_bytes;
      if (g.nd == 0) {
        mbar_arrive_expect_tx(&mbar_d[ps], 0);
        return;
      }
      const uint8_t* blob = slot_blob(ps);
      const Span a = span_of(blob + p.lay.down_q + (size_t)g.ja * g.qbi, (uint32_t)(g.nd * g.qbi));
      const Span b = span_of(blob + p.lay.down_sb + (size_t)g.ja * g.sbbi, (uint32_t)(g.nd * g.sbbi));
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      mbar_arrive_expect_tx(&mbar_d[ps], a.len + b.len);
      bulk_g2s(buf, a.src, a.len, &mbar_d[ps]);
      bulk_g2s(buf + p.d_cap_q, b.src, b.len, &mbar_d[ps]);
    };
    // job order per slot: its gate/up chunks, then the previous slot's down rows
    auto pump = [&](uint32_t limit) {
      while (pr_slot <= NS) {
        if (pr_slot == NS) {
          if (NS - 1 >= p.S && !pr_routed) return;
          issue_d(NS - 1);
          ++pr_slot;
          return;
        }
        if (pr_slot >= p.S && !pr_routed) return;
        if (pr_chunk < g.nch) {
          if (g_issue >= limit) return;
          issue_gu(pr_slot, pr_chunk);
          ++pr_chunk;
          continue;
        }
        if (pr_slot >= 1) issue_d(pr_slot - 1);
        ++pr_slot;
        pr_chunk = 0;
      }
    };

    // ---- prologue ----
    if (tid == 0) {
      pr_slot = 0;
      pr_chunk = 0;
      pr_routed = false;
      pump(g_cons + p.nstage);          // shared-expert rows need no routing
    }
    const float* hin = p.norm ? (l == 0 ? p.out : p.hbuf + (size_t)((l - 1) & 1) * H) : p.x;
    const float* res = p.norm ? hin : p.residual;
    float* outp = p.norm ? ((l == p.L - 1 && !p.copy_back) ? p.out : p.hbuf + (size_t)(l & 1) * H) : p.out;

    if (tid < 32) {
      int id; float w;
      warp_route(p.logits + (size_t)l * p.E, p.E, p.K, id, w);
      if (lane < p.K) {
        s_ids[p.S + lane] = id;
        s_w[p.S + lane] = w;
        if (c == 0 && p.ids_out != nullptr) {
          p.ids_out[(size_t)l * p.K + lane] = id;
          p.w_out[(size_t)l * p.K + lane] = w;
        }
      }
    }
    {
      float ss = 0.f, wg = 0.f;
      for (int e = tid * 4; e < H; e += kFusedThreads * 4) {
        const float4 v = p.norm ? __ldcg(reinterpret_cast<const float4*>(hin + e))
                                : __ldg(reinterpret_cast<const float4*>(hin + e));
        ss += (v.x * v.x + v.y * v.y) + (v.z * v.z + v.w * v.w);
        if (p.S) {
          const uint2 wb = __ldg(reinterpret_cast<const uint2*>(lp.wsg + e));
          wg += (bf16lo(wb.x) * v.x + bf16hi(wb.x) * v.y) + (bf16lo(wb.y) * v.z + bf16hi(wb.y) * v.w);
        }
      }
      ss = warp_sum(ss);
      wg = warp_sum(wg);
      if (lane == 0) {
        s_red[2 * (tid >> 5)] = ss;
        s_red[2 * (tid >> 5) + 1] = wg;
      }
    }
    __syncthreads();
    float SS = 0.f, WG = 0.f;
#pragma unroll
    for (int w = 0; w < kFusedThreads / 32; ++w) {
      SS += s_red[2 * w];
      WG += s_red[2 * w + 1];
    }
    const float rinv = p.norm ? 1.0f / sqrtf(SS / (float)H + p.eps) : 1.0f;
    const float gate = p.S ? sigmoid_f(WG * rinv) : 0.f;
    if (tid == 0 && p.S) {
      s_ids[0] = -1;
      s_w[0] = gate;
      if (c == 0 && p.gate_out != nullptr) p.gate_out[l] = gate;
    } else if (tid == 0 && c == 0 && p.gate_out != nullptr) {
      p.gate_out[l] = 0.f;
    }
    float xs[kSlice];
    float xsum;
    if (p.norm) xsum = load_slice_x<BITS, true>(hin, g.sl, rinv, xs);
    else xsum = load_slice_x<BITS, false>(hin, g.sl, 1.0f, xs);
    __syncthreads();
    if (tid == 0) {
      pr_routed = true;
      pump(g_cons + p.nstage);
    }
#pragma unroll
    for (int i = 0; i < kMaxRowsPerTeam; ++i) accd[i] = 0.f;

    // ---- down rows of one slot, folded into the accumulators ----
    auto do_down = [&](int ps) {
      if (tid == 0) wait_counter(&ctr[ps], (uint32_t)n, p.timeout_ns, p.err);
      mbar_wait(&mbar_d[ps], (uint32_t)(l & 1), p.timeout_ns, p.err);
      __syncthreads();
      float hs[kSlice];
      const float hsum = load_slice_x<BITS, true>(p.hmid + (size_t)hidx(ps) * I, g.dsl, 1.0f, hs);
      const float wk = s_w[ps];
      const uint8_t* buf = darea + (size_t)ps * p.dslot_bytes;
      const uint8_t* q0 = buf + span_off((size_t)g.ja * g.qbi);
      const uint8_t* sb0 = buf + p.d_cap_q + span_off((size_t)g.ja * g.sbbi);
#pragma unroll
      for (int i = 0; i < kMaxRowsPerTeam; ++i) {
        const int jj = g.dteam + i * g.teams_d;
        if (jj < g.nd) {
          SliceCodes<BITS> q;
          if constexpr (BITS == 4) q.v = *reinterpret_cast<const uint4*>(q0 + (size_t)jj * g.qbi + g.dsl * 16);
          else q.v = *reinterpret_cast<const uint2*>(q0 + (size_t)jj * g.qbi + g.dsl * 8);
          const uint32_t sbw = *reinterpret_cast<const uint32_t*>(sb0 + (size_t)jj * g.sbbi + (g.dsl >> 1) * 4);
          accd[i] = fmaf(wk, slice_term<BITS>(q, sbw, hs, hsum), accd[i]);
        }
      }
    };

    // ---- gate/up stream ----
    for (int ps = 0; ps < NS; ++ps) {
      for (int pc = 0; pc < g.nch; ++pc) {
        const uint32_t st = g_cons % p.nstage;
        mbar_wait(&mbar_ring[st], (g_cons / p.nstage) & 1u, p.timeout_ns, p.err);
        const int r0 = g.ra + pc * g.teams_gu;
        const int rn = min(g.teams_gu, g.ra + g.nr - r0);
        const uint8_t* buf = ring + (size_t)st * p.stage_bytes;
        float ga = 0.f, ua = 0.f;
        if (g.team < rn) {
          const uint8_t* gq = buf + span_off((size_t)r0 * g.qbh) + (size_t)g.team * g.qbh;
          const uint8_t* gsb = buf + p.gu_cap_q + span_off((size_t)r0 * g.sbbh) + (size_t)g.team * g.sbbh;
          const uint8_t* uq = buf + p.gu_cap_q + p.gu_cap_sb + span_off((size_t)r0 * g.qbh) + (size_t)g.team * g.qbh;
          const uint8_t* usb =
              buf + 2 * p.gu_cap_q + p.gu_cap_sb + span_off((size_t)r0 * g.sbbh) + (size_t)g.team * g.sbbh;
          SliceCodes<BITS> qg, qu;
          if constexpr (BITS == 4) {
            qg.v = *reinterpret_cast<const uint4*>(gq + g.sl * 16);
            qu.v = *reinterpret_cast<const uint4*>(uq + g.sl * 16);
          } else {
            qg.v = *reinterpret_cast<const uint2*>(gq + g.sl * 8);
            qu.v = *reinterpret_cast<const uint2*>(uq + g.sl * 8);
          }
          const uint32_t sg = *reinterpret_cast<const uint32_t*>(gsb + (g.sl >> 1) * 4);
          const uint32_t su = *reinterpret_cast<const uint32_t*>(usb + (g.sl >> 1) * 4);
          ga = slice_term<BITS>(qg, sg, xs, xsum);
          ua = slice_term<BITS>(qu, su, xs, xsum);
        }
        // team reduction of (ga, ua): split the pair at half width, then fold
        {
          const int half = g.red_w >> 1;
          const bool low = (lane & half) == 0;
          const float send = low ? ua : ga;
          const float recv = __shfl_xor_sync(0xFFFFFFFFu, send, half);
          float v = (low ? ga : ua) + recv;
          for (int o = half >> 1; o >= 1; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
          const int pos = lane & (g.red_w - 1);
          if (g.team < rn && (pos == 0 || pos == half)) {
            float* dst = s_part + ((((g_cons & 1u) * 32 + g.team) * 2 + (pos == 0 ? 0 : 1)) * 8 + g.wit);
            *dst = v;
          }
        }
        __syncthreads();
        if (tid < rn) {
          const float* src = s_part + (((g_cons & 1u) * 32 + tid) * 2) * 8;
          float a = 0.f, u = 0.f;
          for (int w = 0; w < g.wpt; ++w) {
            a += src[w];
            u += src[8 + w];
          }
          p.hmid[(size_t)hidx(ps) * I + r0 + tid] = silu_f(a) * u;
        }
        ++g_cons;
        if (tid == 0) pump(g_cons + p.nstage);
      }
      __syncthreads();
      if (tid == 0) signal_counter(&ctr[ps]);
      if (ps >= 1) do_down(ps - 1);
    }
    do_down(NS - 1);

    // ---- combine + residual, written by each row's owner ----
#pragma unroll
    for (int i = 0; i < kMaxRowsPerTeam; ++i) {
      const int jj = g.dteam + i * g.teams_d;
      const float v = warp_sum(accd[i], g.tl_d);
      if (g.dsl == 0 && jj < g.nd) {
        const int j = g.ja + jj;
        const float r = p.norm ? __ldcg(res + j) : res[j];
        outp[j] = r + v;
      }
    }

    if (l < p.L - 1 || p.copy_back) {
      __syncthreads();
      if (tid == 0) {
        signal_counter(&ctr[NS]);
        wait_counter(&ctr[NS], (uint32_t)n, p.timeout_ns, p.err);
      }
      __syncthreads();
    }
  }

  if (p.copy_back) {
    for (int j = g.ja + tid; j < g.ja + g.nd; j += kFusedThreads) p.out[j] = __ldcg(p.hbuf + j);
  }

  // the last block out resets the counters for the next launch
  __syncthreads();
  if (tid == 0) {
    uint32_t* exit_ctr = p.counters + (size_t)p.L * (NS + 1);
    __threadfence();
    const uint32_t old = atomicAdd(exit_ctr, 1u);
    if (old == (uint32_t)n - 1) {
      for (int i = 0; i < p.L * (NS + 1); ++i) p.counters[i] = 0;
      *exit_ctr = 0;
      __threadfence();
    }
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
static bool pow2(int v) { return v > 0 && (v & (v - 1)) == 0; }

FusedPlan fused_plan(int bits, int H, int I, int K, int S, int device) {
  FusedPlan pl{};
  pl.ok = false;
  const int tl_gu = H / kSlice, tl_d = I / kSlice;
  if (H % kSlice || I % kSlice || !pow2(tl_gu) || !pow2(tl_d)) return pl;
  if (tl_gu < 2 || tl_gu > kFusedThreads || tl_d < 1 || tl_d > 32) return pl;
  if (K + S > kMaxSlots) return pl;
  int sms = 0, smem_max = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) return pl;
  if (cudaDeviceGetAttribute(&smem_max, cudaDevAttrMaxSharedMemoryPerBlockOptin, device) != cudaSuccess) return pl;
  const int grid = sms;
  const int teams_gu = kFusedThreads / tl_gu, teams_d = kFusedThreads / tl_d;
  const int ndmax = (H + grid - 1) / grid;
  if ((ndmax + teams_d - 1) / teams_d > kMaxRowsPerTeam) return pl;
  if (teams_gu > 32) return pl;
  const size_t qbh = (size_t)H * bits / 8, sbbh = (size_t)H / kGroup * 4;
  const size_t qbi = (size_t)I * bits / 8, sbbi = (size_t)I / kGroup * 4;
  pl.gu_cap_q = (int)round_up(teams_gu * qbh + 16, 16);
  pl.gu_cap_sb = (int)round_up(teams_gu * sbbh + 32, 16);
  pl.stage_bytes = (int)round_up(2 * (pl.gu_cap_q + pl.gu_cap_sb), 128);
  pl.d_cap_q = (int)round_up(ndmax * qbi + 16, 16);
  pl.d_cap_sb = (int)round_up(ndmax * sbbi + 32, 16);
  pl.dslot_bytes = (int)round_up(pl.d_cap_q + pl.d_cap_sb, 128);
  const long long avail = (long long)smem_max - kCtrlBytes - (long long)(K + S) * pl.dslot_bytes;
  const long long ns = avail / pl.stage_bytes;
  if (ns < 2) return pl;
  pl.nstage = (int)(ns > kMaxStages ? kMaxStages : ns);
  pl.smem = (size_t)kCtrlBytes + (size_t)pl.nstage * pl.stage_bytes + (size_t)(K + S) * pl.dslot_bytes;
  pl.grid = grid;
  pl.ok = true;
  return pl;
}

template <int BITS>
static cudaError_t launch_fused_t(FusedParams& p, const FusedPlan& pl, cudaStream_t st) {
  static int configured_smem = -1;
  cudaError_t e;
  if (configured_smem < (int)pl.smem) {
    e = cudaFuncSetAttribute(fused_moe_kernel<BITS>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pl.smem);
    if (e != cudaSuccess) return e;
    configured_smem = (int)pl.smem;
  }
  static size_t checked_smem = 0;
  if (checked_smem != pl.smem) {
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fused_moe_kernel<BITS>, kFusedThreads, pl.smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorCooperativeLaunchTooLarge;
    checked_smem = pl.smem;
  }
  // cooperative: all blocks resident at once (the per-slot and per-layer
  // counters are waited on by every block)
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
  p.nstage = pl.nstage;
  p.stage_bytes = pl.stage_bytes;
  p.dslot_bytes = pl.dslot_bytes;
  p.gu_cap_q = pl.gu_cap_q;
  p.gu_cap_sb = pl.gu_cap_sb;
  p.d_cap_q = pl.d_cap_q;
  p.d_cap_sb = pl.d_cap_sb;
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
