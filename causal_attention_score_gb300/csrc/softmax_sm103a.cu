// Fused causal softmax of the score rows on sm_103a:
//
//   att[b][h][t][t2] = exp(s - m) / sum_{u <= t} exp(s_u - m)   for t2 <= t,
//   att[b][h][t][t2] = 0                                          for t2 > t,
//   s = (Q[b][h][t][:] . K[b][h][t2][:]) / sqrt(HS),  m = max_{u <= t} s_u,
//
// the scores of "llm.c dev/cuda/trimat_forward.cu" (trimul_cpu, whose comment
// says it is taken from the attention forward pass) followed by the two-pass
// row softmax of the "Smallem" article 5 (row maximum and sum of exponentials,
// then normalisation). The scores never reach global memory.
//
// Design (one persistent launch, one CTA per SM, 11 warps):
//  - work unit = one (b, h) row block of 128 query rows; units are taken from
//    a per-launch counter, longest row blocks first.
//  - warp 0: TMA producer. Per unit it loads the Q tile once (two buffers, so
//    the next unit's Q arrives while this one computes) and streams the unit's
//    K tiles j = 0..i twice through a multi-stage ring.
//  - warp 1: tcgen05.mma issuer, 128 x 128 x HS per tile into one of two TMEM
//    accumulators, both passes.
//  - warps 2..9: epilogue, each owning 32 rows x 64 columns of every tile.
//    Pass 1 keeps, per row, the running maximum m and sum l of exp2 of the
//    scores (log2 domain); the two warps holding the two halves of a row then
//    combine (m, l) through shared memory behind a bounded mbarrier. Pass 2
//    recomputes each tile and writes exp2((x - m) - log2 l) (the maximum and
//    the log-sum kept apart, as the article does), staged through swizzled
//    shared memory into 32 x 32 TMA stores (plain stores when T % 4 != 0).
//  - warp 10: writes the tiles above the diagonal (probability 0) from a global
//    pool of 128 x 128 zero tiles, as 128 x 16 TMA stores of a zeroed shared
//    buffer (plain stores when T % 4 != 0). It takes a tile only while its own
//    epilogue is not storing (start-up, pass 1, after the last unit), two tiles
//    in flight at most, and no more than its share of the pool: (Tt - 1) /
//    (Tt + 1) zero tiles per pass-1 tile its epilogue has started (Tt = tiles
//    per row), plus a slack of two, until the epilogue has no more units. So
//    the SM's write stream has no gaps, and the pool lasts into the second half
//    of the launch and evens out its end across SMs.
//  - Writes saturate HBM and queue ahead of reads, so the producer prefetches
//    the next unit's Q and first K tiles into L2 a whole unit early; K is kept
//    in L2 (every row block of its (b, h) reads it, twice), the output is not.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <string>

#include "csa_internal.h"
#include "sm103a_ptx.cuh"

namespace csa {
namespace {

constexpr int kTile = 128;
constexpr int kChunkElems = 64;
constexpr int kChunkBytes = kTile * 128;
constexpr int kEpiWarps = 8;
constexpr int kZeroWarp = 2 + kEpiWarps;
constexpr int kThreads = 64 + 32 * kEpiWarps + 32;
constexpr int kSlabCols = 64;
constexpr int kBoxBytes = 32 * 32 * 4;
constexpr int kPairBytes = 2 * kBoxBytes;  // one 32 x 64 fp32 slab as two TMA boxes
constexpr int kZeroCols = 128, kZeroRows = 16;  // zero-writer TMA box
constexpr int kZeroBytes = kZeroCols * kZeroRows * 4;
constexpr int kStatsBytes = 2 * kEpiWarps * 32 * 8;  // (m, l) per row half, two units
constexpr int kTmemCols = 2 * kTile;
constexpr int kRingDepth = 4;
constexpr unsigned int kEnd = 0xFFFFFFFFu;
constexpr uint32_t kIdesc = idesc_bf16_f32(kTile, kTile);

// Work-list counters: [0] row-block units, [1] finished CTAs, [2] zero tiles; sets
// handed out by acquire_counter_slot (one per stream, or one per captured launch).
// The last CTA to finish resets its set.
constexpr int kSchedWords = kCounterWords;
__device__ unsigned int g_softmax_sched[kDirectSlots + kCaptureSlots][kSchedWords];
constexpr int kPrefetchK = 4;  // K tiles of the next unit prefetched into L2
// Staging pairs per epilogue warp (at most) and K ring depth (at most).
#ifndef CSA_SOFTMAX_MAX_PAIRS
#define CSA_SOFTMAX_MAX_PAIRS 1
#endif
#ifndef CSA_SOFTMAX_MAX_STAGES
#define CSA_SOFTMAX_MAX_STAGES 8
#endif
#ifndef CSA_SOFTMAX_ZERO_PACE
#define CSA_SOFTMAX_ZERO_PACE 1
#endif
constexpr bool kZeroPace = CSA_SOFTMAX_ZERO_PACE != 0;  // pace the zero writer (zero_share_q16)
constexpr uint32_t kZeroSlack = 2;                      // zero tiles ahead of the share

struct SoftmaxArgs {
  int T, NH, BH, Tt;
  int kchunks, ksteps, stages;
  int n_units;
  int n_zero;  // zero tiles: BH * Tt * (Tt - 1) / 2
  // Zero tiles per computed (lower) tile, 16.16 fixed point: a CTA's zero writer
  // keeps its count within this share of the pass-1 tiles its epilogue has
  // started (plus kZeroSlack), so the pool lasts through the launch instead of
  // running dry while the later units' pass 1 leaves the SM with nothing to store.
  uint32_t zero_share_q16;
  float scale_log2e;  // log2(e) / sqrt(HS)
  uint32_t tma_store;
  uint32_t pairs;  // staging pairs per epilogue warp (1 or 2)
  float* out;
  int* status;
  unsigned long long wait_limit_ns;
  unsigned int* sched;
  unsigned long long* done;  // completion word of the counter set
  unsigned long long seq;    // written there by the last CTA, after the counters' reset
  int inject;  // withhold each CTA's first Q load (watchdog tests)
  uint32_t q_bytes, k_bytes;
  uint32_t off_k, off_staging, off_zero, off_stats, off_bars, off_misc;
};

// Unit p: row block i = Tt - 1 - p / BH (longest first) of (b, h) = p % BH.
__device__ __forceinline__ void decode_unit(unsigned int p, const SoftmaxArgs& a, int& bh,
                                            int& ti) {
  const int row = static_cast<int>(p) / a.BH;
  bh = static_cast<int>(p) - row * a.BH;
  ti = a.Tt - 1 - row;
}

__global__ void __launch_bounds__(kThreads, 1)
    softmax_sm103a_kernel(const __grid_constant__ CUtensorMap tmap_qkv,
                          const __grid_constant__ CUtensorMap tmap_out,
                          const __grid_constant__ CUtensorMap tmap_zero, const SoftmaxArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);

  const uint32_t warp = threadIdx.x >> 5;
  const uint32_t lane = lane_id();
  const int S = a.stages;

  const uint32_t bars = base + a.off_bars;
  auto qfull_bar = [&](int s) { return bars + 8u * s; };
  auto qempty_bar = [&](int s) { return bars + 8u * (2 + s); };
  auto kfull_bar = [&](int s) { return bars + 8u * (4 + s); };
  auto kempty_bar = [&](int s) { return bars + 8u * (4 + S + s); };
  auto tfull_bar = [&](int s) { return bars + 8u * (4 + 2 * S + s); };
  auto tempty_bar = [&](int s) { return bars + 8u * (6 + 2 * S + s); };
  const uint32_t drain_bar = bars + 8u * (8 + 2 * S);
  // Row statistics exchange of the two warps that share TMEM lane quarter p (the
  // two 64-column halves of the same rows): one barrier per pair.
  auto stats_bar = [&](uint32_t p) { return bars + 8u * (10 + 2 * S + 2 * kRingDepth + p); };
  auto rfull_bar = [&](int s) { return bars + 8u * (10 + 2 * S + s); };
  auto rempty_bar = [&](int s) { return bars + 8u * (10 + 2 * S + kRingDepth + s); };
  const uint32_t tmem_slot = base + a.off_misc;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + a.off_misc + 4);
  // Set while the epilogue is in pass 2 (storing), read by the zero writer.
  volatile int* epi_storing = reinterpret_cast<volatile int*>(gbase + a.off_misc + 8);
  auto ring_entry = [&](int s) { return base + a.off_misc + 16u + 4u * s; };
  // Pass-1 tiles the epilogue has started, and set once it has no more units
  // (the zero writer's pacing; see zero_share_q16).
  volatile int* p1_started =
      reinterpret_cast<volatile int*>(gbase + a.off_misc + 16u + 4u * kRingDepth);
  volatile int* epi_done =
      reinterpret_cast<volatile int*>(gbase + a.off_misc + 20u + 4u * kRingDepth);
  auto q_chunk = [&](int qb, int kc) { return base + qb * a.q_bytes + kc * kChunkBytes; };
  auto k_chunk = [&](int s, int kc) { return base + a.off_k + s * a.k_bytes + kc * kChunkBytes; };
  const uint32_t stats = base + a.off_stats;
  const uint32_t zero_buf = base + a.off_zero;

  const Watchdog wd{a.wait_limit_ns, a.status, abort_flag};

  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(qfull_bar(s), 1);
      mbar_init(qempty_bar(s), 1);
      mbar_init(tfull_bar(s), 1);
      mbar_init(tempty_bar(s), kEpiWarps);
    }
    for (int s = 0; s < S; ++s) {
      mbar_init(kfull_bar(s), 1);
      mbar_init(kempty_bar(s), 1);
    }
    mbar_init(drain_bar, 1);
    for (uint32_t p = 0; p < 4; ++p) mbar_init(stats_bar(p), 2);
    for (int s = 0; s < kRingDepth; ++s) {
      mbar_init(rfull_bar(s), 1);
      mbar_init(rempty_bar(s), 1 + kEpiWarps);
    }
    *abort_flag = 0;
    *epi_storing = 0;
    *p1_started = 0;
    *epi_done = 0;
    fence_barrier_init();
  }
  if (a.tma_store) {
    for (uint32_t w = threadIdx.x; w < kZeroBytes / 16; w += kThreads)
      st_shared_v4(zero_buf + 16u * w, 0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
    tc_fence_before_sync();
  }
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = ld_shared_b32(tmem_slot);

  // Nothing global has been touched yet: the kernel ahead in the stream may still
  // be running (programmatic launch), so wait for it here.
  grid_dependency_wait();

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer --
    if (lane == 0) {
      tma_prefetch_map(&tmap_qkv);
      int stage = 0, qb = 0, slot = 0;
      uint32_t phase = 0, qphase = 0, sphase = 0;
      uint32_t kissued = 0, kparity = 0, qissued = 0, qparity = 0;
      const uint32_t qtx = a.q_bytes, ktx = a.k_bytes;
      const uint64_t keep = l2_policy_evict_last(), once = l2_policy_evict_first();
      // Prefetches unit p's Q and K tiles into L2 (nothing past the work list).
      auto prefetch_unit = [&](unsigned int p) {
        if (p >= static_cast<unsigned int>(a.n_units)) return;
        int pbh, pti;
        decode_unit(p, a, pbh, pti);
        const int pb = pbh / a.NH, ph = pbh - pb * a.NH;
        for (int kc = 0; kc < a.kchunks; ++kc) {
          tma_prefetch_l2_4d(&tmap_qkv, kc * kChunkElems, ph, pti * kTile, pb, keep);
          for (int tj = 0; tj <= pti && tj < kPrefetchK; ++tj)
            tma_prefetch_l2_4d(&tmap_qkv, kc * kChunkElems, a.NH + ph, tj * kTile, pb, keep);
        }
      };
      unsigned int p0 = atomicAdd(a.sched, 1u), p1 = atomicAdd(a.sched, 1u);
      prefetch_unit(p1);
      bool ok = true, injected = false;
      while (ok) {
        const unsigned int cur = p0;
        const bool done = cur >= static_cast<unsigned int>(a.n_units);
        p0 = p1;
        if (!done) {
          p1 = atomicAdd(a.sched, 1u);
          prefetch_unit(p1);
        }
        if (!mbar_wait(rempty_bar(slot), sphase ^ 1u, wd, kSiteSched)) break;
        st_shared_b32(ring_entry(slot), done ? kEnd : cur);
        mbar_arrive(rfull_bar(slot));
        if (++slot == kRingDepth) {
          slot = 0;
          sphase ^= 1u;
        }
        if (done) break;
        int bh, ti;
        decode_unit(cur, a, bh, ti);
        if (!CSA_CHECK(bh >= 0 && bh < a.BH && ti >= 0 && ti < a.Tt, wd, kCheckTile)) break;
        const int b = bh / a.NH, h = bh - b * a.NH;
        if (!mbar_wait(qempty_bar(qb), qphase ^ 1u, wd, kSiteProducerEmpty)) break;
        mbar_arrive_expect_tx(qfull_bar(qb), qtx);
        if (a.inject && !injected) {
          injected = true;  // withhold this CTA's first Q tile: the MMA warp's wait must run out
          qissued &= ~(1u << qb);
        } else {
          for (int kc = 0; kc < a.kchunks; ++kc)
            tma_load_4d_hint(q_chunk(qb, kc), &tmap_qkv, qfull_bar(qb), kc * kChunkElems, h,
                             ti * kTile, b, once);
          qissued |= 1u << qb;
          qparity = (qparity & ~(1u << qb)) | (qphase << qb);
        }
        if (++qb == 2) {
          qb = 0;
          qphase ^= 1u;
        }
        for (int pass = 0; ok && pass < 2; ++pass) {
          for (int tj = 0; tj <= ti; ++tj) {
            if (!mbar_wait(kempty_bar(stage), phase ^ 1u, wd, kSiteProducerEmpty)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(kfull_bar(stage), ktx);
            for (int kc = 0; kc < a.kchunks; ++kc)
              tma_load_4d_hint(k_chunk(stage, kc), &tmap_qkv, kfull_bar(stage), kc * kChunkElems,
                               a.NH + h, tj * kTile, b, keep);
            kissued |= 1u << stage;
            kparity = (kparity & ~(1u << stage)) | (phase << stage);
            if (++stage == S) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
      if (*abort_flag) {
        // Let every load still in flight land before shared memory goes away.
        for (int s = 0; s < S + 2; ++s) {
          const bool is_q = s >= S;
          const int i = is_q ? s - S : s;
          if (!((is_q ? qissued : kissued) & (1u << i))) continue;
          const uint32_t bar = is_q ? qfull_bar(i) : kfull_bar(i);
          const uint32_t par = ((is_q ? qparity : kparity) >> i) & 1u;
          const uint64_t t0 = globaltimer_ns();
          while (!mbar_test(bar, par) && globaltimer_ns() - t0 < a.wait_limit_ns) {
          }
        }
      }
    }
  } else if (warp == 1) {
    // -------------------------------------------------------- MMA issuer --
    if (lane == 0) {
      int stage = 0, qb = 0, acc = 0, slot = 0;
      uint32_t phase = 0, qphase = 0, acc_phase = 0, sphase = 0;
      bool ok = true;
      while (ok) {
        if (!mbar_wait(rfull_bar(slot), sphase, wd, kSiteSched)) break;
        const unsigned int cur = ld_shared_b32(ring_entry(slot));
        mbar_arrive(rempty_bar(slot));
        if (++slot == kRingDepth) {
          slot = 0;
          sphase ^= 1u;
        }
        if (cur == kEnd) break;
        int bh, ti;
        decode_unit(cur, a, bh, ti);
        if (!mbar_wait(qfull_bar(qb), qphase, wd, kSiteMmaFull)) break;
        tc_fence_after_sync();
        for (int pass = 0; ok && pass < 2; ++pass) {
          for (int tj = 0; tj <= ti; ++tj) {
            if (!mbar_wait(tempty_bar(acc), acc_phase ^ 1u, wd, kSiteMmaTmemEmpty) ||
                !mbar_wait(kfull_bar(stage), phase, wd, kSiteMmaFull)) {
              ok = false;
              break;
            }
            tc_fence_after_sync();
            if (!CSA_CHECK(acc >= 0 && (acc + 1) * kTile <= kTmemCols, wd, kCheckTmem)) {
              ok = false;
              break;
            }
            const uint32_t d = tmem_base + static_cast<uint32_t>(acc * kTile);
            for (int k = 0; k < a.ksteps; ++k) {
              const uint32_t off = static_cast<uint32_t>(k & 3) * 32u;
              umma_bf16(d, umma_desc_k_sw128(q_chunk(qb, k >> 2) + off),
                        umma_desc_k_sw128(k_chunk(stage, k >> 2) + off), kIdesc,
                        k > 0 ? 1u : 0u);
            }
            umma_commit(kempty_bar(stage));
            umma_commit(tfull_bar(acc));
            if (++stage == S) {
              stage = 0;
              phase ^= 1u;
            }
            if (++acc == 2) {
              acc = 0;
              acc_phase ^= 1u;
            }
          }
        }
        if (!ok) break;
        umma_commit(qempty_bar(qb));  // the unit's MMAs are done with its Q tile
        if (++qb == 2) {
          qb = 0;
          qphase ^= 1u;
        }
      }
      umma_commit(drain_bar);
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_test(drain_bar, 0) && globaltimer_ns() - t0 < a.wait_limit_ns) {
      }
    }
  } else if (warp == kZeroWarp) {
    // ------------------------------------------------------- zero writer --
    // Columns c >= (i + 1) * 128 of row block i hold probability 0 whatever the
    // row statistics are; this warp writes them with streaming stores while the
    // epilogue computes, so they never queue in front of its TMA stores.
    const int T = a.T;
    const bool vec = a.tma_store != 0;  // T % 4 == 0 and a 16-byte aligned output
    const uint64_t once = l2_policy_evict_first();
    const int Tt = a.Tt;
    int taken = 0;
    bool ok = true;
    while (ok) {
      // Yield to the epilogue while it stores, and keep within this CTA's share of
      // zero tiles until its epilogue has no more units (bounded: the epilogue
      // leaves pass 2, starts a unit or finishes within the wait limit, or the
      // CTA aborts).
      int z = 0;
      if (lane == 0) {
        const uint64_t t0 = globaltimer_ns();
        auto hold = [&]() {
          if (*epi_storing != 0) return true;
          if (!kZeroPace || *epi_done != 0) return false;
          const uint32_t quota = static_cast<uint32_t>(
              (static_cast<unsigned long long>(*p1_started) * a.zero_share_q16) >> 16);
          return static_cast<uint32_t>(taken) >= quota + kZeroSlack;
        };
        for (uint32_t it = 0; hold(); ++it) {
          if (*abort_flag) {
            ok = false;
            break;
          }
          if ((it & 63u) == 63u && globaltimer_ns() - t0 > a.wait_limit_ns) {
            *abort_flag = 1;
            if (atomicCAS(a.status, 0, CSA_ERR_TIMEOUT) == 0) atomicExch(a.status + 1, kSiteSched);
            ok = false;
            break;
          }
          __nanosleep(128);
        }
        z = ok ? static_cast<int>(atomicAdd(a.sched + 2, 1u)) : a.n_zero;
      }
      z = __shfl_sync(0xffffffffu, z, 0);
      if (z >= a.n_zero) break;
      ++taken;
      // Zero tile z: (b, h) = z % BH, then the strictly upper tile (i, j), j > i,
      // numbered by pairing block rows i and Tt - 2 - i (Tt tiles per pair).
      const int w = z / a.BH;
      const int bh = z - w * a.BH;
      const int pr = w / Tt, o = w - pr * Tt;
      if (!CSA_CHECK(bh >= 0 && bh < a.BH && pr >= 0 && pr < Tt, wd, kCheckTile)) break;
      int ti, tj;
      if (o < Tt - 1 - pr) {
        ti = pr;
        tj = pr + 1 + o;
      } else {
        ti = Tt - 2 - pr;
        tj = ti + 1 + (o - (Tt - 1 - pr));
      }
      const int r0 = ti * kTile, c0 = tj * kTile;  // rows r0.. are all < T (ti <= Tt - 2)
      if (vec) {
        if (lane == 0) {
          // Columns past T - 1 are clipped by the tensor map.
          for (int rr = 0; rr < kTile; rr += kZeroRows)
            tma_store_3d_hint(&tmap_zero, zero_buf, c0, r0 + rr, bh, once);
          bulk_commit();
          bulk_wait_read<1>();  // two tiles in flight at most
        }
        __syncwarp();
      } else {
        const int cols = min(kTile, T - c0);
        float* blk = a.out + (static_cast<size_t>(bh) * T + r0) * T + c0;
        for (int rr = 0; rr < kTile; ++rr)
          for (int i = static_cast<int>(lane); i < cols; i += 32)
            blk[static_cast<size_t>(rr) * T + i] = 0.0f;
      }
    }
    // Only the stores' reads of shared memory must finish before the CTA exits;
    // their global writes complete before the grid does.
    if (lane == 0) bulk_wait_read<0>();
    __syncwarp();
  } else {
    // ---------------------------------------------------------- epilogue --
    // Warp ew = warp - 2 owns the 32 rows of TMEM lane quarter warp % 4 and the
    // 64-column slab ew / 4 of every tile; warp ew ^ 4 holds the other half of
    // the same rows.
    const uint32_t ew = warp - 2u;
    const int q = static_cast<int>(warp & 3u);
    const int slab = static_cast<int>(ew >> 2);
    const uint32_t staging = base + a.off_staging + ew * a.pairs * kPairBytes;
    uint32_t pair = 0;
    const int T = a.T;
    const uint64_t once = l2_policy_evict_first();
    int acc = 0, slot = 0;
    uint32_t acc_phase = 0, sphase = 0, stats_phase = 0;
    bool ok = true;
    while (ok) {
      int got = 1;
      unsigned int cur = 0;
      if (lane == 0) {
        got = mbar_wait(rfull_bar(slot), sphase, wd, kSiteSched) ? 1 : 0;
        if (got) {
          cur = ld_shared_b32(ring_entry(slot));
          mbar_arrive(rempty_bar(slot));
        }
      }
      got = __shfl_sync(0xffffffffu, got, 0);
      cur = __shfl_sync(0xffffffffu, cur, 0);
      if (!got || cur == kEnd) break;
      if (++slot == kRingDepth) {
        slot = 0;
        sphase ^= 1u;
      }
      int bh, ti;
      decode_unit(cur, a, bh, ti);
      if (!CSA_CHECK(bh >= 0 && bh < a.BH && ti >= 0 && ti < a.Tt, wd, kCheckTile)) break;
      if (ew == 0 && lane == 0) *p1_started = *p1_started + ti + 1;
      const int row0 = ti * kTile + q * 32;
      const int r = row0 + static_cast<int>(lane);
      // The unit's 2n tiles (pass 1: tj = 0..ti, then pass 2 over the same tiles)
      // come out of the accumulators in order. The TMEM load of tile k + 1 is
      // issued before tile k is processed, so its latency hides behind the
      // arithmetic; exactly one load is outstanding whenever a buffer is in use.
      const int n = ti + 1;
      const float sc = a.scale_log2e;
      float m = -INFINITY, l = 0.0f, lg = 0.0f;
      uint32_t va[kSlabCols], vb[kSlabCols];
      int held = 0;
      auto issue = [&](uint32_t(&v)[kSlabCols]) -> bool {
        if (!mbar_wait_warp_inline(tfull_bar(acc), acc_phase, wd, kSiteEpilogueFull)) return false;
        tc_fence_after_sync();
        tmem_ld_64cols_async(tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                 static_cast<uint32_t>(acc * kTile + slab * kSlabCols),
                             v);
        held = acc;
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
        return true;
      };
      auto retire = [&](uint32_t(&v)[kSlabCols]) {
        tmem_wait_ld_64(v);
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(tempty_bar(held));
      };
      auto process = [&](uint32_t(&v)[kSlabCols], int k) -> bool {
        const bool second = k >= n;
        const int tj = second ? k - n : k;
        const int colw = tj * kTile + slab * kSlabCols;
        // Columns of this slab in row r's causal window are the offsets e <= lim.
        const int lim = min(r, T - 1) - colw;
        // Lane 0 has the warp's smallest window, so this test is warp-uniform.
        const bool full = min(row0, T - 1) - colw >= kSlabCols - 1;
        if (!second) {
          // The maximum is taken on the raw products; scaling by sc > 0 is
          // monotone in fp32, so it commutes with the maximum.
          float mx = -INFINITY;
          if (full) {
            float t[kSlabCols / 2];
#pragma unroll
            for (int e = 0; e < kSlabCols / 2; ++e)
              t[e] = fmaxf(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1]));
#pragma unroll
            for (int w = kSlabCols / 4; w >= 1; w >>= 1)
#pragma unroll
              for (int e = 0; e < w; ++e) t[e] = fmaxf(t[e], t[e + w]);
            mx = t[0];
          } else {
#pragma unroll
            for (int e = 0; e < kSlabCols; ++e)
              if (e <= lim) mx = fmaxf(mx, __uint_as_float(v[e]));
          }
          mx *= sc;
          if (mx > m) {
            l *= ex2_approx(m - mx);
            m = mx;
          }
          float part[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) part[e] = 0.0f;
          if (full) {
            // Pairs of columns through the packed fp32 pipe: x * sc - m, then the
            // partial sums, two lanes per instruction.
            const uint64_t sc2 = pack_f32x2(sc, sc), nm2 = pack_f32x2(-m, -m);
            uint64_t p2[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) p2[j] = 0ull;
#pragma unroll
            for (int e = 0; e < kSlabCols; e += 2) {
              float t0, t1;
              fma_f32x2(t0, t1, __uint_as_float(v[e]), __uint_as_float(v[e + 1]), sc2, nm2);
              p2[(e >> 1) & 3] = add_f32x2(p2[(e >> 1) & 3], pack_f32x2(ex2_approx(t0), ex2_approx(t1)));
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) unpack_f32x2(p2[j], part[2 * j], part[2 * j + 1]);
          } else {
#pragma unroll
            for (int e = 0; e < kSlabCols; ++e)
              if (e <= lim) part[e & 7] += ex2_approx(fmaf(__uint_as_float(v[e]), sc, -m));
          }
          l += ((part[0] + part[1]) + (part[2] + part[3])) +
               ((part[4] + part[5]) + (part[6] + part[7]));
          if (k != n - 1) return true;
          // Combine the two halves of each row: (m, l) of this warp and of warp
          // ew ^ 4. Slots alternate between units: a warp can be one unit ahead
          // of its partner's read, never two (that needs the partner's next arrival).
          const uint32_t sbase = stats + stats_phase * (kEpiWarps * 32u * 8u);
          st_shared_b32(sbase + (ew * 32u + lane) * 8u, __float_as_uint(m));
          st_shared_b32(sbase + (ew * 32u + lane) * 8u + 4u, __float_as_uint(l));
          __syncwarp();
          if (lane == 0) mbar_arrive(stats_bar(static_cast<uint32_t>(q)));
          if (!mbar_wait_warp_inline(stats_bar(static_cast<uint32_t>(q)), stats_phase, wd,
                                     kSiteEpilogueFull))
            return false;
          stats_phase ^= 1u;
          const uint32_t other = sbase + ((ew ^ 4u) * 32u + lane) * 8u;
          const float m2 = __uint_as_float(ld_shared_b32(other));
          const float l2 = __uint_as_float(ld_shared_b32(other + 4u));
          const float mm = fmaxf(m, m2);
          const float ll = (m == -INFINITY ? 0.0f : l * ex2_approx(m - mm)) +
                           (m2 == -INFINITY ? 0.0f : l2 * ex2_approx(m2 - mm));
          // Pass 2 writes exp2((x - m) - log2 l): the maximum is subtracted first
          // and log2 l kept apart from it, since folding the two into one number
          // loses log2 l's low bits when the maximum is large.
          m = mm;
          lg = log2f(ll);
          if (ew == 0 && lane == 0) *epi_storing = 1;
          return true;
        }
        if (full) {
          const uint64_t sc2 = pack_f32x2(sc, sc), nm2 = pack_f32x2(-m, -m);
          const uint64_t nl2 = pack_f32x2(-lg, -lg);
#pragma unroll
          for (int e = 0; e < kSlabCols; e += 2) {
            float t0, t1;
            fma_f32x2(t0, t1, __uint_as_float(v[e]), __uint_as_float(v[e + 1]), sc2, nm2);
            float u0, u1;
            unpack_f32x2(add_f32x2(pack_f32x2(t0, t1), nl2), u0, u1);
            v[e] = __float_as_uint(ex2_approx(u0));
            v[e + 1] = __float_as_uint(ex2_approx(u1));
          }
        } else {
#pragma unroll
          for (int e = 0; e < kSlabCols; ++e)
            v[e] = e <= lim ? __float_as_uint(ex2_approx(fmaf(__uint_as_float(v[e]), sc, -m) - lg))
                            : 0u;
        }
        if (row0 >= T || colw >= T) return true;
        if (lane == 0) {
          if (a.pairs == 2) bulk_wait_read<1>();
          else bulk_wait_read<0>();
        }
        __syncwarp();
        const uint32_t box0 = staging + pair * kPairBytes;
        if (++pair == a.pairs) pair = 0;
        const int nbox = (colw + 32 < T) ? 2 : 1;
#pragma unroll
        for (int c = 0; c < 2; ++c)
          if (c < nbox) stage_row_sw128(box0 + c * kBoxBytes, lane, v + 32 * c);
        if (a.tma_store) {
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            for (int c = 0; c < nbox; ++c)
              tma_store_3d_hint(&tmap_out, box0 + c * kBoxBytes, colw + c * 32, row0, bh, once);
            bulk_commit();
          }
        } else {
          __syncwarp();
          for (int c = 0; c < nbox; ++c) {
            const int col = colw + c * 32 + static_cast<int>(lane);
            float* ocol = a.out + (static_cast<size_t>(bh) * T + row0) * T + col;
            for (int rr = 0; rr < 32; ++rr) {
              const uint32_t val =
                  staged_elem_sw128(box0 + c * kBoxBytes, static_cast<uint32_t>(rr), lane);
              if (row0 + rr < T && col < T) ocol[static_cast<size_t>(rr) * T] = __uint_as_float(val);
            }
          }
        }
        return true;
      };
      if (!issue(va)) {
        ok = false;
        break;
      }
      // 2n is even: tiles k (buffer va) and k + 1 (buffer vb) per step.
      for (int k = 0; k < 2 * n; k += 2) {
        retire(va);
        if (!issue(vb)) {
          ok = false;
          break;
        }
        if (!process(va, k)) {
          retire(vb);
          ok = false;
          break;
        }
        retire(vb);
        const bool more = k + 2 < 2 * n;
        if (more && !issue(va)) {
          ok = false;
          break;
        }
        if (!process(vb, k + 1)) {
          if (more) retire(va);
          ok = false;
          break;
        }
      }
      if (ew == 0 && lane == 0) *epi_storing = 0;
      if (!ok) break;
    }
    if (ew == 0 && lane == 0) {
      *epi_storing = 0;
      *epi_done = 1;
    }
    // Only the stores' reads of shared memory must finish before the CTA exits;
    // their global writes complete before the grid does.
    if (lane == 0) bulk_wait_read<0>();
    __syncwarp();
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, kTmemCols);
  }
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(a.sched + 1, 1u) == gridDim.x - 1) {
      atomicExch(a.sched, 0u);
      atomicExch(a.sched + 2, 0u);
      atomicExch(a.sched + 1, 0u);
      if (a.done) {
        // the set is free for another stream once the host sees this
        __threadfence_system();
        *reinterpret_cast<volatile unsigned long long*>(a.done) = a.seq;
      }
    }
  }
}

}  // namespace

int softmax_launch(float* out, const void* qkv, int B, int T, int C, int NH, cudaStream_t stream,
                   const DeviceInfo& dev, std::string& err) {
  const int HS = C / NH;
  if (HS % 8 != 0) {
    err = "causal_softmax_forward: HS = C/NH must be a multiple of 8";
    return CSA_ERR_ALIGN;
  }
  if (HS > 128) {
    err = "causal_softmax_forward: HS > 128 is not supported";
    return CSA_ERR_UNSUPPORTED;
  }
  if (reinterpret_cast<uintptr_t>(qkv) % 16 != 0 || reinterpret_cast<uintptr_t>(out) % 4 != 0) {
    err = "causal_softmax_forward: qkv must be 16-byte aligned and out 4-byte aligned";
    return CSA_ERR_ALIGN;
  }
  const long long BH = static_cast<long long>(B) * NH;
  const long long Tt = (static_cast<long long>(T) + kTile - 1) / kTile;
  if (BH * Tt * (Tt - 1) / 2 >= (1LL << 31) - (1LL << 20) || BH * Tt >= (1LL << 31) - (1LL << 20) ||
      BH > (1LL << 30)) {
    err = "causal_softmax_forward: too many tiles";
    return CSA_ERR_SHAPE;
  }
  SoftmaxArgs a{};
  a.T = T;
  a.NH = NH;
  a.BH = static_cast<int>(BH);
  a.Tt = static_cast<int>(Tt);
  a.kchunks = (HS + kChunkElems - 1) / kChunkElems;
  a.ksteps = (HS + 15) / 16;
  a.n_units = static_cast<int>(BH * Tt);
  a.n_zero = static_cast<int>(BH * Tt * (Tt - 1) / 2);
  a.zero_share_q16 = static_cast<uint32_t>((static_cast<unsigned long long>(Tt - 1) << 16) /
                                           static_cast<unsigned long long>(Tt + 1));
  a.scale_log2e = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(HS)));
  a.tma_store = (T % 4 == 0 && reinterpret_cast<uintptr_t>(out) % 16 == 0) ? 1u : 0u;
  a.out = out;
  a.status = dev.status_word;
  a.wait_limit_ns = wait_limit_ns();
  a.inject = take_inject() ? 1 : 0;

  // Shared memory: Q (2 buffers) | K ring | staging | zero box | stats | barriers | misc.
  a.q_bytes = static_cast<uint32_t>(a.kchunks) * kChunkBytes;
  a.k_bytes = a.q_bytes;
  // The most staging pairs per epilogue warp (up to CSA_SOFTMAX_MAX_PAIRS) that
  // still leave two K stages; the rest of shared memory deepens the K ring.
  int staging_bytes = 0;
  for (int pairs = CSA_SOFTMAX_MAX_PAIRS; pairs >= 1; --pairs) {
    staging_bytes = kEpiWarps * pairs * kPairBytes;
    const int fixed = 2 * static_cast<int>(a.q_bytes) + staging_bytes + kZeroBytes + kStatsBytes +
                      1024 + 1024;
    a.pairs = static_cast<uint32_t>(pairs);
    a.stages = std::min(CSA_SOFTMAX_MAX_STAGES, (dev.max_smem_optin - fixed) / static_cast<int>(a.k_bytes));
    if (a.stages >= 2) break;
  }
  if (a.stages < 2) {
    err = "causal_softmax_forward: not enough shared memory";
    return CSA_ERR_UNSUPPORTED;
  }
  a.off_k = 2u * a.q_bytes;
  a.off_staging = a.off_k + static_cast<uint32_t>(a.stages) * a.k_bytes;
  a.off_zero = a.off_staging + static_cast<uint32_t>(staging_bytes);
  a.off_stats = a.off_zero + kZeroBytes;
  a.off_bars = a.off_stats + kStatsBytes;
  a.off_misc = a.off_bars + 8u * static_cast<uint32_t>(10 + 2 * a.stages + 2 * kRingDepth + 4);
  const size_t smem = a.off_misc + 16 + 4 * kRingDepth + 8 + 1024;

  CUtensorMap map_qkv, map_out, map_zero;
  {
    const uint64_t dims[4] = {static_cast<uint64_t>(HS), static_cast<uint64_t>(3 * NH),
                              static_cast<uint64_t>(T), static_cast<uint64_t>(B)};
    const uint64_t strides[3] = {static_cast<uint64_t>(HS) * 2, static_cast<uint64_t>(C) * 6,
                                 static_cast<uint64_t>(T) * C * 6};
    const uint32_t box[4] = {kChunkElems, 1, kTile, 1};
    int rc = encode_tiled(&map_qkv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, qkv, dims, strides, box,
                          CU_TENSOR_MAP_SWIZZLE_128B, err);
    if (rc != CSA_OK) return rc;
  }
  if (a.tma_store) {
    const uint64_t dims[3] = {static_cast<uint64_t>(T), static_cast<uint64_t>(T),
                              static_cast<uint64_t>(BH)};
    const uint64_t strides[2] = {static_cast<uint64_t>(T) * 4,
                                 static_cast<uint64_t>(T) * static_cast<uint64_t>(T) * 4};
    const uint32_t box[3] = {32, 32, 1};
    int rc = encode_tiled(&map_out, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, out, dims, strides, box,
                          CU_TENSOR_MAP_SWIZZLE_128B, err);
    if (rc != CSA_OK) return rc;
    const uint32_t zbox[3] = {kZeroCols, kZeroRows, 1};
    rc = encode_tiled(&map_zero, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, out, dims, strides, zbox,
                      CU_TENSOR_MAP_SWIZZLE_NONE, err);
    if (rc != CSA_OK) return rc;
  } else {
    std::memset(&map_out, 0, sizeof map_out);
    std::memset(&map_zero, 0, sizeof map_zero);
  }
  {
    int rc = set_max_dynamic_smem(reinterpret_cast<const void*>(softmax_sm103a_kernel),
                                  static_cast<int>(smem), dev.device, err);
    if (rc != CSA_OK) {
      err = "causal_softmax_forward: " + err;
      return rc;
    }
  }
  CounterSlot slot;
  {
    static std::mutex mu;
    static unsigned int* sched_base[64] = {};
    {
      std::lock_guard<std::mutex> lock(mu);
      if (dev.device < 0 || dev.device >= 64) {
        err = "causal_softmax_forward: device ordinal out of range";
        return CSA_ERR_CUDA;
      }
      if (!sched_base[dev.device]) {
        void* p = nullptr;
        cudaError_t se = cudaGetSymbolAddress(&p, g_softmax_sched);
        if (se != cudaSuccess) {
          err = std::string("causal_softmax_forward: cudaGetSymbolAddress: ") +
                cudaGetErrorString(se);
          return CSA_ERR_CUDA;
        }
        sched_base[dev.device] = static_cast<unsigned int*>(p);
      }
    }
    int rc = acquire_counter_slot(kFamilySoftmax, dev, sched_base[dev.device], stream, slot, err);
    if (rc != CSA_OK) {
      err = "causal_softmax_forward: " + err;
      return rc;
    }
    a.sched = slot.counters;
    a.done = slot.done;
    a.seq = slot.seq;
  }
  cudaError_t e;
  const long long grid = std::min<long long>(a.n_units, dev.sm_count);
  e = launch_programmatic(softmax_sm103a_kernel, static_cast<unsigned>(grid), kThreads, smem,
                          stream, map_qkv, map_out, map_zero, a);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) {
    abandon_counter_slot(kFamilySoftmax, dev, slot);
    err = std::string("causal_softmax_forward: launch: ") + cudaGetErrorString(e);
    return CSA_ERR_LAUNCH;
  }
  return CSA_OK;
}

}  // namespace csa
