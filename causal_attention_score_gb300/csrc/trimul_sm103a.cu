// Causal triangular score product on sm_103a.
//
//   out[b][h][t][t2] = (Q[b][h][t][:] . K[b][h][t2][:]) * (1/sqrt(HS))  for t2 <= t
//   out[b][h][t][t2] = mask                                            for t2 > t
//
// as defined by the CPU referee of "llm.c dev/cuda/trimat_forward.cu"
// (trimul_cpu, Chapter I), reading Q and K in place from the packed
// (B, T, 3, NH, HS) tensor (trimul_global's q/k pointers, Chapter II) with no
// permute pass.
//
// Design (one persistent launch, one CTA per SM, 11 warps):
//  - tile space: for every (b, h) the ceil(T/128)^2 output tiles of 128 x 128;
//    tiles with t2-tile <= t-tile are "lower" (MMA + epilogue), the others are
//    "fill" tiles that only receive the mask pattern (not written at all in
//    lower-only mode). The lower tiles form the work list that the producer,
//    MMA and epilogue warps walk; the fill tiles form a separate launch-wide
//    pool (warp 10). With fill tiles, CTAs take work-list positions from a
//    per-launch counter; otherwise (lower-only, the batched NT product) they
//    are dealt statically and the counters are never touched.
//  - warp 0 (one lane): TMA producer. A 4-D tensor map (HS, 3*NH, T, B) over
//    the packed QKV addresses the query of head h at index h and its key at
//    NH + h; rows past T and columns past HS arrive zero-filled. Q and K tiles
//    land in a multi-stage ring in the 128-byte-swizzled K-major layout.
//  - warp 1 (one lane): tcgen05.mma issuer, M=128 N=128 K=16, bf16 x bf16 ->
//    fp32 into one of two TMEM accumulators (256 columns), so the epilogue of
//    one tile overlaps the MMA of the next.
//  - warps 2..9: epilogue. Each warp owns 32 rows (its TMEM lane quarter) and
//    64 columns: tcgen05.ld, multiply by 1/sqrt(HS), write the mask above the
//    diagonal on diagonal tiles, stage through swizzled shared memory and
//    issue 32 x 32 TMA stores (clipped at T). When T % 4 != 0 the output rows
//    are not 16-byte aligned, so the same staged data is written with
//    coalesced plain stores. In lower-only mode the 32 x 32 boxes that straddle
//    the diagonal are written by each lane from registers, its row's t2 <= t
//    part only.
//  - fp32 inputs ("kind::tf32" form, trimul_forward_f32): the referee's own
//    input type, computed to fp32 accuracy with three tf32 products: each
//    input x splits exactly into hi = x with its low 13 mantissa bits cleared
//    (a tf32 value) and lo = x - hi (an fp32 value; its tf32 rounding costs
//    2^-21 |x|), and each tile accumulates hi.hi + hi.lo + lo.hi (lo.lo is
//    below 2^-20 |q.k|). The tensor core reads only the top 19 bits of an fp32
//    operand, so the loaded x serves as hi as it is (measured: bit-identical
//    results to explicitly cleared operands). With HS <= 128 the Q tile of a
//    row block lives in TMEM as the MMA's A operand: its hi and lo parts take
//    2 * HS of the 512 columns beside the two accumulators, written once per
//    row block by warps 11-14 (one per lane quarter, tcgen05.st) from Q
//    chunks that pass through the ring (two such Q buffers when HS <= 64, so
//    the next row block's Q is written while the current one is in use). The
//    ring then carries only K, one raw 32-element chunk per stage; the same
//    warps split each into a three-slot ring of lo parts, and each CTA walks
//    one contiguous run of the work list so that consecutive tiles share their
//    Q. In full mode that path is its own instance with one staging box per
//    epilogue warp, which leaves room for more ring stages. With
//    128 < HS <= 256 a stage holds one 32-element chunk of both Q and K and
//    their lo parts.
//  - warp 10: fill writer. It takes fill tiles from the launch-wide pool while
//    the epilogue has nothing to store (start-up, a wait on the MMA, after the
//    last lower tile) and writes each as 128 x 16 TMA stores of a resident
//    mask buffer, two tiles in flight at most. The operand loads queue behind
//    the launch's writes in the memory system, so the epilogue stalls now and
//    then; the fills keep the SM's write stream going meanwhile, and the pool
//    evens out the end of the launch across SMs.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <mutex>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <string>

#include "csa_internal.h"
#include "sm103a_ptx.cuh"

namespace csa {
namespace {

constexpr int kTile = 128;          // output tile edge
constexpr int kChunkElems = 64;     // bf16 per 128-byte swizzle row
constexpr int kChunkElemsF32 = 32;  // fp32 per 128-byte swizzle row
constexpr int kChunkBytes = kTile * 128;  // one 128-row x 64-element operand chunk
// Tuning constants (compile-time): operand ring depth and staging box pairs per
// epilogue warp; the host picks the deepest staging that still leaves two stages.
#ifndef CSA_TRIMUL_MAX_STAGES
#define CSA_TRIMUL_MAX_STAGES 4
#endif
#ifndef CSA_TRIMUL_MAX_STORE_GROUPS
#define CSA_TRIMUL_MAX_STORE_GROUPS 1
#endif
// fp32 form with Q in TMEM: raw-chunk ring depth and K lo ring slots.
#ifndef CSA_TRIMUL_MAX_STAGES_QT
#define CSA_TRIMUL_MAX_STAGES_QT 8
#endif
#ifndef CSA_TRIMUL_LO_SLOTS
#define CSA_TRIMUL_LO_SLOTS 3
#endif
// fp32 form with Q in TMEM: one staging box per epilogue warp (1) or a pair (0).
#ifndef CSA_TRIMUL_F32_SINGLE_BOX
#define CSA_TRIMUL_F32_SINGLE_BOX 1
#endif
// fp32 form with Q in TMEM: Q buffers when two fit (1 or 2).
#ifndef CSA_TRIMUL_Q_BUFS
#define CSA_TRIMUL_Q_BUFS 2
#endif

constexpr int kEpiWarps = 8;        // two per TMEM lane quarter
constexpr int kFillWarp = 2 + kEpiWarps;
constexpr int kThreads = 64 + 32 * kEpiWarps + 32;
constexpr int kConvWarps = 4;  // fp32 form: warps 11-14 split each stage into hi and lo
constexpr int kFirstConvWarp = kFillWarp + 1;
constexpr int kThreadsF32 = kThreads + 32 * kConvWarps;
constexpr int kFillCols = 128, kFillRows = 16;  // fill-writer TMA box
constexpr int kFillBytes = kFillCols * kFillRows * 4;
constexpr int kSlabCols = 64;       // accumulator columns per epilogue warp
constexpr int kBoxBytes = 32 * 32 * 4;  // one 32 x 32 fp32 TMA store box
constexpr int kTmemCols = 2 * kTile;
constexpr uint32_t kIdesc = idesc_bf16_f32(kTile, kTile);
constexpr uint32_t kIdescTf32 = idesc_tf32_f32(kTile, kTile);

struct TrimulArgs {
  int T, T2, BH, Tt, Tt2;  // rows / columns of each (b, h) output and their tile counts
  int nh_div, b_off;       // operand coordinates: A (bh % nh_div), B (b_off + bh % nh_div),
                           // both at outer index bh / nh_div
  uint32_t causal;         // 1: triangular tiles, mask above the diagonal; 0: all tiles
  int kchunks, ksteps, stages;
  int n_lower;  // tiles with t2-tile <= t-tile (all tiles when not causal): the work list
  int n_fill;   // tiles with t2-tile > t-tile: the fill pool (0 in lower-only mode)
  int per_lower, per_fill;  // lower / fill tiles per (b, h)
  uint32_t dynamic;     // 1: work-list positions from the shared counter; 0: dealt statically
  unsigned int* sched;  // this launch's counters: [0] next position, [1] CTAs done, [2] next fill
  unsigned long long* done;  // completion word of the counter set (nullptr: none)
  unsigned long long seq;    // written there by the last CTA, after the counters' reset
  float scale;
  uint32_t mask_bits;
  uint32_t lower_only;
  uint32_t tma_store;
  float* out;
  int* status;
  unsigned long long wait_limit_ns;
  int inject;
  uint32_t store_groups;  // staging box pairs per epilogue warp (1 or 2; 0: a single box)
  uint32_t staging_stride;  // staging bytes per epilogue warp
  uint32_t stage_bytes, off_staging, off_mask, off_bars, off_misc;
  // Operand chunks (128-byte rows) per stage, and stages per tile: bf16 keeps a
  // whole tile's chunks in one stage; the fp32 form streams one chunk per stage.
  int stage_chunks, tile_stages, chunk_elems;
  // fp32 form with HS <= 128: Q's hi / lo parts held in TMEM (the MMA's A
  // operand) for a whole row block; a ring stage then holds one K chunk and
  // its lo part, or a Q chunk on its way to TMEM.
  uint32_t q_tmem;
  uint32_t contig;  // static deal as one contiguous run of the work list per CTA
  int tmem_cols;    // TMEM columns allocated: 256, or 512 with q_tmem
  // With q_tmem the ring holds raw chunks only; the lo parts of K chunks go to
  // a separate ring of lo_slots chunks at off_lo, freed by the MMA's commit.
  int lo_slots;
  uint32_t off_lo;
  // Q buffers in TMEM (1, or 2 when two fit: HS <= 64), so that the next row
  // block's Q is written while the MMAs still read the current one.
  int q_bufs;
};

// Counters per launch: [0] work-list position, [1] finished CTAs, [2] fill tile.
constexpr int kSchedWords = kCounterWords;

// Work-list counter sets, handed out by acquire_counter_slot (one per stream, or
// one per captured launch); the last CTA of a launch resets its set to zero.
__device__ unsigned int g_trimul_sched[kDirectSlots + kCaptureSlots][kSchedWords];

#ifndef CSA_TRIMUL_SCHED_DEPTH
#define CSA_TRIMUL_SCHED_DEPTH 4
#endif
#ifndef CSA_TRIMUL_FETCH_AHEAD
#define CSA_TRIMUL_FETCH_AHEAD 2
#endif
constexpr int kSchedDepth = CSA_TRIMUL_SCHED_DEPTH;  // positions buffered between roles
constexpr int kFetchAhead = CSA_TRIMUL_FETCH_AHEAD;  // work-list fetches in flight (1..4)
constexpr unsigned int kEntryEnd = 0xFFFFFFFFu;      // ring entry: no more work

// Position p of the work list: (b, h) = p / per_lower, so CTAs working at the
// same time share Q and K tiles in L2; r = p % per_lower is the tile's number
// among the (b, h)'s computed tiles.
__device__ __forceinline__ void decode_position(int p, int per_lower, int& bh, int& r) {
  bh = p / per_lower;
  r = p - bh * per_lower;
}

// Largest i with i * (i + 1) / 2 <= r.
__device__ __forceinline__ int tri_root(int r) {
  int i = static_cast<int>((sqrtf(8.0f * static_cast<float>(r) + 1.0f) - 1.0f) * 0.5f);
  while ((i + 1) * (i + 2) / 2 <= r) ++i;
  while (i * (i + 1) / 2 > r) --i;
  return i;
}

// Lower tile number r (j <= i) of one (b, h), row block by row block.
__device__ __forceinline__ void decode_lower(int r, int& ti, int& tj) {
  ti = tri_root(r);
  tj = r - ti * (ti + 1) / 2;
}

// Computed tile number r of one (b, h): the lower triangle in causal mode, row
// by row over all Tt2 column tiles otherwise.
__device__ __forceinline__ void decode_computed(int r, uint32_t causal, int Tt2, int& ti,
                                                int& tj) {
  if (causal) {
    decode_lower(r, ti, tj);
  } else {
    ti = r / Tt2;
    tj = r - ti * Tt2;
  }
}

// Fill tile number r (j > i) of one (b, h): the transpose of the strictly-lower
// enumeration.
__device__ __forceinline__ void decode_fill(int r, int& ti, int& tj) {
  const int i = tri_root(r) + 1;  // i * (i - 1) / 2 <= r < i * (i + 1) / 2
  ti = r - i * (i - 1) / 2;       // row tile (smaller index)
  tj = i;                         // column tile
}

// kSingleBox (fp32 with Q in TMEM, full mode): one staging box per epilogue warp
// instead of a pair, so the operand rings get 32 KB more shared memory. A
// separate instance: the lower-only fp32 form measured 16 % slower with this
// path merely compiled into its kernel.
template <bool kF32, bool kSingleBox = false>
__global__ void __launch_bounds__(kF32 ? kThreadsF32 : kThreads, 1)
    trimul_sm103a_kernel(const __grid_constant__ CUtensorMap tmap_a,
                         const __grid_constant__ CUtensorMap tmap_b,
                         const __grid_constant__ CUtensorMap tmap_out,
                         const __grid_constant__ CUtensorMap tmap_fill, const TrimulArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);

  const uint32_t warp = threadIdx.x >> 5;
  const uint32_t lane = lane_id();

  const uint32_t bars = base + a.off_bars;
  auto full_bar = [&](int s) { return bars + 8u * s; };
  auto empty_bar = [&](int s) { return bars + 8u * (a.stages + s); };
  auto tfull_bar = [&](int s) { return bars + 8u * (2 * a.stages + s); };
  auto tempty_bar = [&](int s) { return bars + 8u * (2 * a.stages + 2 + s); };
  const uint32_t drain_bar = bars + 8u * (2 * a.stages + 4);
  auto sfull_bar = [&](int s) { return bars + 8u * (2 * a.stages + 5 + s); };
  auto sempty_bar = [&](int s) { return bars + 8u * (2 * a.stages + 5 + kSchedDepth + s); };
  // fp32 form: stage s split into hi / lo and ready for the MMA.
  auto conv_bar = [&](int s) { return bars + 8u * (2 * a.stages + 5 + 2 * kSchedDepth + s); };
  // Q in TMEM: the MMAs reading the Q in buffer b are complete (it may be replaced).
  auto qfree_bar = [&](uint32_t b) { return bars + 8u * (3 * a.stages + 5 + 2 * kSchedDepth + b); };
  // Q in TMEM: lo slot l of the K lo ring is free again.
  auto lofree_bar = [&](int l) { return bars + 8u * (3 * a.stages + 7 + 2 * kSchedDepth + l); };
  auto lo_slot = [&](int l) { return base + a.off_lo + static_cast<uint32_t>(l) * kChunkBytes; };
  constexpr int kBlockThreads = kF32 ? kThreadsF32 : kThreads;
  auto sched_entry = [&](int s) { return base + a.off_misc + 16u + 4u * s; };
  const uint32_t tmem_slot = base + a.off_misc;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + a.off_misc + 4);
  // Set while the epilogue has nothing to store; the fill writer works then.
  volatile int* epi_idle = reinterpret_cast<volatile int*>(gbase + a.off_misc + 8);
  const uint32_t mask_box = base + a.off_mask;
  auto q_chunk = [&](int s, int kc) { return base + s * a.stage_bytes + kc * kChunkBytes; };
  auto k_chunk = [&](int s, int kc) {
    return base + s * a.stage_bytes + (a.stage_chunks + kc) * kChunkBytes;
  };
  // fp32 form without Q in TMEM: the lo parts of a stage's Q and K chunks
  // follow its raw chunks.
  auto lo_chunk = [&](uint32_t hi) { return hi + 2u * kChunkBytes; };
  // Q in TMEM: columns of buffer b's hi and lo parts (after the two accumulators).
  const uint32_t q_cols = 32u * static_cast<uint32_t>(a.kchunks);
  auto qhi_col = [&](uint32_t b) { return kTmemCols + 2u * q_cols * b; };
  auto qlo_col = [&](uint32_t b) { return kTmemCols + 2u * q_cols * b + q_cols; };

  const Watchdog wd{a.wait_limit_ns, a.status, abort_flag};

  if (threadIdx.x == 0) {
    for (int s = 0; s < a.stages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(tfull_bar(s), 1);
      mbar_init(tempty_bar(s), kEpiWarps);
    }
    mbar_init(drain_bar, 1);
    for (int s = 0; s < kSchedDepth; ++s) {
      mbar_init(sfull_bar(s), 1);
      mbar_init(sempty_bar(s), 1 + kEpiWarps + (kF32 ? kConvWarps : 0));
    }
    if (kF32) {
      for (int s = 0; s < a.stages; ++s) mbar_init(conv_bar(s), kConvWarps);
      mbar_init(qfree_bar(0), 1);
      mbar_init(qfree_bar(1), 1);
      for (int l = 0; l < a.lo_slots; ++l) mbar_init(lofree_bar(l), 1);
    }
    *abort_flag = 0;
    *epi_idle = 1;
    fence_barrier_init();
  }
  // The resident mask buffer that fill tiles are stored from.
  if (a.n_fill > 0 && a.tma_store) {
    for (uint32_t w = threadIdx.x; w < kFillBytes / 4; w += kBlockThreads)
      st_shared_b32(mask_box + 4u * w, a.mask_bits);
    fence_proxy_async_smem();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, static_cast<uint32_t>(a.tmem_cols));
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
      tma_prefetch_map(&tmap_a);
      tma_prefetch_map(&tmap_b);
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0, issued_parity = 0;  // per-stage: loads that may be in flight
      bool injected = false;
      // Bytes per stage: one chunk with Q in TMEM (a K chunk, or a Q chunk on its
      // way to TMEM), else the stage's Q and K chunks.
      const uint32_t tx = a.q_tmem ? static_cast<uint32_t>(kChunkBytes)
                                   : static_cast<uint32_t>(a.stage_chunks) * 2u * kChunkBytes;
      // Work list: the computed tiles, (b, h)-major. Positions are taken from a
      // shared counter (kFetchAhead fetches in flight) when a fill pool absorbs
      // the imbalance that leaves, else dealt statically (c, c+G, ...) so that
      // every CTA knows its operands ahead. Each position goes to the MMA and
      // epilogue warps through the shared ring.
      const bool dynamic = a.dynamic != 0;
      // Static deals: c, c+G, c+2G, ...; or (contig) the run [c*n/G, (c+1)*n/G),
      // whose consecutive tiles mostly share a row block.
      const long long n_lower = a.n_lower;
      unsigned int static_next =
          a.contig ? static_cast<unsigned int>(blockIdx.x * n_lower / gridDim.x) : blockIdx.x;
      const unsigned int static_end =
          static_cast<unsigned int>((blockIdx.x + 1ll) * n_lower / gridDim.x);
      auto fetch = [&]() -> unsigned int {
        if (dynamic) return atomicAdd(a.sched, 1u);
        if (kF32 && a.contig)
          return static_next < static_end ? static_next++ : static_cast<unsigned int>(a.n_lower);
        const unsigned int v = static_next;
        static_next += gridDim.x;
        return v;
      };
      int q_bh = -1, q_ti = -1;  // the row block whose Q is in TMEM
      const uint64_t l2_keep = l2_policy_evict_last(), l2_once = l2_policy_evict_first();
      unsigned int pf[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) pf[i] = i < kFetchAhead ? fetch() : 0u;
      int slot = 0;
      uint32_t sphase = 0;
      while (true) {
        const unsigned int cur = pf[0];
        const bool done = cur >= static_cast<unsigned int>(a.n_lower);
#pragma unroll
        for (int i = 0; i < 3; ++i) pf[i] = pf[i + 1];
        if (!done) pf[kFetchAhead - 1] = fetch();
        if (!mbar_wait(sempty_bar(slot), sphase ^ 1u, wd, kSiteSched)) break;
        st_shared_b32(sched_entry(slot), done ? kEntryEnd : cur);
        mbar_arrive(sfull_bar(slot));
        if (++slot == kSchedDepth) {
          slot = 0;
          sphase ^= 1u;
        }
        if (done) break;
        int bh, r, ti, tj;
        decode_position(static_cast<int>(cur), a.per_lower, bh, r);
        decode_computed(r, a.causal, a.Tt2, ti, tj);
        if (!CSA_CHECK(bh >= 0 && bh < a.BH && ti >= 0 && ti < a.Tt && tj >= 0 && tj < a.Tt2 &&
                           stage >= 0 && stage < a.stages,
                       wd, kCheckTile))
          break;
        const int outer = bh / a.nh_div, inner = bh - outer * a.nh_div;
        // Q in TMEM: a new row block first sends its Q chunks through the ring.
        const bool new_q = kF32 && a.q_tmem && (bh != q_bh || ti != q_ti);
        if (new_q) {
          q_bh = bh;
          q_ti = ti;
        }
        const int q_stages = new_q ? a.kchunks : 0;
        bool ok = true;
        for (int ts = 0; ts < q_stages + a.tile_stages; ++ts) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1u, wd, kSiteProducerEmpty)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(full_bar(stage), tx);
          if (a.inject && !injected) {
            injected = true;  // withhold this CTA's first loads: its consumer's wait must run out
            issued &= ~(1u << stage);
          } else if (kF32 && a.q_tmem) {
            // CTAs walk separate runs of the list here, so a K tile's later uses
            // come from other rows after much output has streamed through L2:
            // K is kept there (evict_last), Q is read once per row block.
            const bool is_q = ts < q_stages;
            const int x = (is_q ? ts : ts - q_stages) * a.chunk_elems;
            if (is_q)
              tma_load_4d_hint(q_chunk(stage, 0), &tmap_a, full_bar(stage), x, inner, ti * kTile,
                               outer, l2_once);
            else
              tma_load_4d_hint(q_chunk(stage, 0), &tmap_b, full_bar(stage), x, a.b_off + inner,
                               tj * kTile, outer, l2_keep);
            issued |= 1u << stage;
            issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
          } else {
            for (int kc = 0; kc < a.stage_chunks; ++kc) {
              const int x = (ts * a.stage_chunks + kc) * a.chunk_elems;
              tma_load_4d(q_chunk(stage, kc), &tmap_a, full_bar(stage), x, inner, ti * kTile,
                          outer);
              tma_load_4d(k_chunk(stage, kc), &tmap_b, full_bar(stage), x, a.b_off + inner,
                          tj * kTile, outer);
            }
            issued |= 1u << stage;
            issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
          }
          if (++stage == a.stages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
      }
      if (*abort_flag) {
        // Let every load still in flight land before shared memory goes away.
        const Watchdog drain{a.wait_limit_ns, a.status, abort_flag};
        for (int s = 0; s < a.stages; ++s) {
          if (!(issued & (1u << s))) continue;
          const uint32_t par = (issued_parity >> s) & 1u;
          const uint64_t t0 = globaltimer_ns();
          while (!mbar_test(full_bar(s), par) && globaltimer_ns() - t0 < drain.limit_ns) {
          }
        }
      }
    }
  } else if (warp == 1) {
    // -------------------------------------------------------- MMA issuer --
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      int slot = 0;
      uint32_t sphase = 0;
      int q_bh = -1, q_ti = -1;  // Q in TMEM: the row block it holds, and how many so far
      uint32_t n_q = 0;
      int lo = 0;         // Q in TMEM: next slot of the K lo ring
      uint32_t qbuf = 0;  // Q in TMEM: the buffer the current Q is in
      while (true) {
        if (!mbar_wait(sfull_bar(slot), sphase, wd, kSiteSched)) break;
        const unsigned int cur = ld_shared_b32(sched_entry(slot));
        mbar_arrive(sempty_bar(slot));
        if (++slot == kSchedDepth) {
          slot = 0;
          sphase ^= 1u;
        }
        if (cur == kEntryEnd) break;
        if constexpr (kF32) {
          if (a.q_tmem) {
            int bh, r, ti, tj;
            decode_position(static_cast<int>(cur), a.per_lower, bh, r);
            decode_computed(r, a.causal, a.Tt2, ti, tj);
            if (bh != q_bh || ti != q_ti) {
              q_bh = bh;
              q_ti = ti;
              // The splitter may overwrite the previous Q's buffer once the MMAs
              // reading it are complete.
              const bool two = a.q_bufs == 2;
              if (n_q > 0) umma_commit(qfree_bar(two ? ((n_q - 1u) & 1u) : 0u));
              qbuf = two ? (n_q & 1u) : 0u;
              ++n_q;
              // The row block's Q chunks: written to TMEM by the splitter, which
              // then hands each ring slot back through this thread.
              bool q_ok = true;
              for (int c = 0; c < a.kchunks; ++c) {
                if (!mbar_wait(conv_bar(stage), phase, wd, kSiteMmaFull)) {
                  q_ok = false;
                  break;
                }
                mbar_arrive(empty_bar(stage));
                if (++stage == a.stages) {
                  stage = 0;
                  phase ^= 1u;
                }
              }
              if (!q_ok) break;
            }
          }
        }
        if (!mbar_wait(tempty_bar(acc), acc_phase ^ 1u, wd, kSiteMmaTmemEmpty)) break;
        tc_fence_after_sync();
        if (!CSA_CHECK(acc >= 0 && (acc + 1) * kTile <= static_cast<int>(a.tmem_cols) &&
                           (!a.q_tmem || qlo_col(qbuf) + q_cols <= a.tmem_cols),
                       wd, kCheckTmem))
          break;
        const uint32_t d = tmem_base + static_cast<uint32_t>(acc * kTile);
        bool ok = true;
        for (int ts = 0; ts < a.tile_stages; ++ts) {
          if (!mbar_wait(kF32 ? conv_bar(stage) : full_bar(stage), phase, wd, kSiteMmaFull)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          if constexpr (kF32) {
            if (a.q_tmem) {
              // One 32-element K chunk against Q's hi / lo columns in TMEM: 4 steps
              // of 8 along K, each hi.hi + hi.lo + lo.hi.
              // Descriptors built once per stage; a step of 8 tf32 along K adds 32 B
              // (2 in the descriptor's address field) and 8 TMEM columns.
              const uint64_t khi = umma_desc_k_sw128(q_chunk(stage, 0));
              const uint64_t klo = umma_desc_k_sw128(lo_slot(lo));
              const uint32_t ahi = tmem_base + qhi_col(qbuf) + static_cast<uint32_t>(ts) * 32u;
              const uint32_t alo = tmem_base + qlo_col(qbuf) + static_cast<uint32_t>(ts) * 32u;
              umma_tf32_ts(d, ahi, khi, kIdescTf32, ts > 0 ? 1u : 0u);
              umma_tf32_ts(d, ahi, klo, kIdescTf32, 1u);
              umma_tf32_ts(d, alo, khi, kIdescTf32, 1u);
#pragma unroll
              for (uint32_t k = 1; k < 4; ++k) {
                umma_tf32_ts(d, ahi + 8u * k, khi + 2u * k, kIdescTf32, 1u);
                umma_tf32_ts(d, ahi + 8u * k, klo + 2u * k, kIdescTf32, 1u);
                umma_tf32_ts(d, alo + 8u * k, khi + 2u * k, kIdescTf32, 1u);
              }
              umma_commit(lofree_bar(lo));  // lo slot read -> the splitter may refill it
              if (++lo == a.lo_slots) lo = 0;
            } else {
            // One 32-element chunk: 4 steps of 8 along K, each hi.hi + hi.lo + lo.hi.
            const uint32_t qh = q_chunk(stage, 0), kh = k_chunk(stage, 0);
            for (int k = 0; k < 4; ++k) {
              const uint32_t off = static_cast<uint32_t>(k) * 32u;  // 8 tf32 = 32 B along K
              const uint64_t qhi = umma_desc_k_sw128(qh + off), khi = umma_desc_k_sw128(kh + off);
              umma_tf32(d, qhi, khi, kIdescTf32, (ts > 0 || k > 0) ? 1u : 0u);
              umma_tf32(d, qhi, umma_desc_k_sw128(lo_chunk(kh) + off), kIdescTf32, 1u);
              umma_tf32(d, umma_desc_k_sw128(lo_chunk(qh) + off), khi, kIdescTf32, 1u);
            }
            }
          } else {
            for (int k = 0; k < a.ksteps; ++k) {
              const uint32_t off = static_cast<uint32_t>(k & 3) * 32u;  // 16 bf16 = 32 B along K
              const uint64_t ad = umma_desc_k_sw128(q_chunk(stage, k >> 2) + off);
              const uint64_t bd = umma_desc_k_sw128(k_chunk(stage, k >> 2) + off);
              umma_bf16(d, ad, bd, kIdesc, k > 0 ? 1u : 0u);
            }
          }
          umma_commit(empty_bar(stage));  // operands consumed -> slot free
          if (++stage == a.stages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(tfull_bar(acc));  // accumulator ready -> epilogue
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      // All MMAs of this thread complete before TMEM can be released.
      umma_commit(drain_bar);
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_test(drain_bar, 0) && globaltimer_ns() - t0 < a.wait_limit_ns) {
      }
    }
  } else if (kF32 && warp >= kFirstConvWarp) {
    // ---------------------------------------------------------- splitter --
    // For every stage of every computed tile (the work ring tells how many):
    // once its fp32 Q and K chunks have landed, store lo = x - hi beside each
    // value x (hi = x with the low 13 mantissa bits cleared, which is what the
    // tensor core reads of x itself), then hand the stage to the MMA warp.
    // With Q in TMEM, the same warps first write each new row block's Q: warp w
    // owns TMEM lane quarter w % 4, i.e. Q rows 32 (w % 4) .. + 31.
    const uint32_t cw = warp - kFirstConvWarp;
    const uint32_t quarter = warp & 3u;
    int stage = 0, slot = 0;
    uint32_t phase = 0, sphase = 0;
    int q_bh = -1, q_ti = -1;
    uint32_t n_q = 0;
    int lo = 0;  // Q in TMEM: next slot of the K lo ring, and its pass parity
    uint32_t lo_phase = 0;
    bool ok = true;
    while (ok) {
      int got = 1;
      unsigned int cur = 0;
      if (lane == 0) {
        got = mbar_wait(sfull_bar(slot), sphase, wd, kSiteSched) ? 1 : 0;
        if (got) {
          cur = ld_shared_b32(sched_entry(slot));
          mbar_arrive(sempty_bar(slot));
        }
      }
      got = __shfl_sync(0xffffffffu, got, 0);
      cur = __shfl_sync(0xffffffffu, cur, 0);
      if (!got || cur == kEntryEnd) break;
      if (++slot == kSchedDepth) {
        slot = 0;
        sphase ^= 1u;
      }
      if (a.q_tmem) {
        int bh, r, ti, tj;
        decode_position(static_cast<int>(cur), a.per_lower, bh, r);
        decode_computed(r, a.causal, a.Tt2, ti, tj);
        if (bh != q_bh || ti != q_ti) {
          q_bh = bh;
          q_ti = ti;
          // Q number n_q goes to buffer n_q % q_bufs, once the MMAs reading the Q
          // that used it before (number n_q - q_bufs) are complete.
          const bool two = a.q_bufs == 2;
          const uint32_t nb = two ? 2u : 1u;
          const uint32_t qb = two ? (n_q & 1u) : 0u;
          const uint32_t par = two ? (((n_q >> 1) - 1u) & 1u) : ((n_q - 1u) & 1u);
          if (n_q >= nb && !mbar_wait_warp(qfree_bar(qb), par, wd, kSiteMmaFull))
            break;
          tc_fence_after_sync();
          ++n_q;
          const uint32_t row = quarter * 32u + lane;  // this lane's Q row and TMEM lane
          const uint32_t lane_addr = tmem_base + ((quarter * 32u) << 16);
          for (int c = 0; c < a.kchunks; ++c) {
            if (!mbar_wait_warp(full_bar(stage), phase, wd, kSiteMmaFull)) {
              ok = false;
              break;
            }
            // Row `row` of the 128-byte-swizzled chunk: 16-byte unit j sits at
            // position j ^ (row % 8).
            const uint32_t rowp = q_chunk(stage, 0) + row * 128u;
            uint32_t hi[32], lo[32];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              uint32_t x[4];
              asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                           : "=r"(x[0]), "=r"(x[1]), "=r"(x[2]), "=r"(x[3])
                           : "r"(rowp + ((static_cast<uint32_t>(j) ^ (row & 7u)) << 4)));
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                hi[4 * j + e] = x[e] & 0xFFFFE000u;
                lo[4 * j + e] = __float_as_uint(__uint_as_float(x[e]) -
                                                __uint_as_float(hi[4 * j + e]));
              }
            }
            tmem_st_32cols(lane_addr + qhi_col(qb) + 32u * static_cast<uint32_t>(c), hi);
            tmem_st_32cols(lane_addr + qlo_col(qb) + 32u * static_cast<uint32_t>(c), lo);
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(conv_bar(stage));
            if (++stage == a.stages) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (!ok) break;
        }
      }
      for (int ts = 0; ts < a.tile_stages; ++ts) {
        if (!mbar_wait_warp(full_bar(stage), phase, wd, kSiteMmaFull)) {
          ok = false;
          break;
        }
        // The stage's raw chunks (K alone with Q in TMEM, else Q and K: 16 or
        // 32 KB contiguous) as 16-byte words over the lanes of the 4 splitter
        // warps, four loads in flight per lane. The lo parts go to the same
        // offsets of the lo ring's next slot (Q in TMEM) or after the raw chunks.
        const uint32_t hi0 = q_chunk(stage, 0);
        uint32_t lo0 = lo_chunk(hi0);
        const uint32_t words = (a.q_tmem ? 1u : 2u) * kChunkBytes / 16u;
        if (a.q_tmem) {
          if (!mbar_wait_warp(lofree_bar(lo), lo_phase ^ 1u, wd, kSiteMmaFull)) {
            ok = false;
            break;
          }
          lo0 = lo_slot(lo);
          if (++lo == a.lo_slots) {
            lo = 0;
            lo_phase ^= 1u;
          }
        }
        for (uint32_t i0 = cw * 32u + lane; i0 < words; i0 += 4u * 32u * kConvWarps) {
          uint32_t x[4][4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const uint32_t addr = hi0 + 16u * (i0 + u * 32u * kConvWarps);
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(x[u][0]), "=r"(x[u][1]), "=r"(x[u][2]), "=r"(x[u][3])
                         : "r"(addr));
          }
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            uint32_t l4[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              l4[e] = __float_as_uint(__uint_as_float(x[u][e]) -
                                      __uint_as_float(x[u][e] & 0xFFFFE000u));
            st_shared_v4(lo0 + 16u * (i0 + u * 32u * kConvWarps), l4[0], l4[1], l4[2], l4[3]);
          }
        }
        fence_proxy_async_smem();  // generic smem writes -> visible to tcgen05.mma
        __syncwarp();
        if (lane == 0) mbar_arrive(conv_bar(stage));
        if (++stage == a.stages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  } else if (warp == kFillWarp) {
    // ------------------------------------------------------- fill writer --
    const int T = a.T, T2 = a.T2;
    const uint64_t once = l2_policy_evict_first();
    // (no fill pool: the pool counter is left untouched)
    bool ok = a.n_fill > 0;
    while (ok) {
      int f = 0;
      if (lane == 0) {
        // Wait (bounded) until the epilogue has nothing to store.
        const uint64_t t0 = globaltimer_ns();
        if (*abort_flag) ok = false;
        for (uint32_t it = 0; ok && *epi_idle == 0; ++it) {
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
          __nanosleep(64);
        }
        f = ok ? static_cast<int>(atomicAdd(a.sched + 2, 1u)) : a.n_fill;
      }
      f = __shfl_sync(0xffffffffu, f, 0);
      if (f >= a.n_fill) break;
      const int bh = f / a.per_fill;
      int ti, tj;
      decode_fill(f - bh * a.per_fill, ti, tj);
      if (!CSA_CHECK(bh < a.BH && ti >= 0 && ti < tj && tj < a.Tt, wd, kCheckTile)) break;
      const int r0 = ti * kTile, c0 = tj * kTile;  // rows r0.. are all < T (ti < tj)
      if (a.tma_store) {
        if (lane == 0) {
          // Columns past T2 - 1 are clipped by the tensor map.
          for (int rr = 0; rr < kTile; rr += kFillRows)
            tma_store_3d_hint(&tmap_fill, mask_box, c0, r0 + rr, bh, once);
          bulk_commit();
          bulk_wait_read<1>();  // two tiles in flight at most
        }
        __syncwarp();
      } else {
        const float m = __uint_as_float(a.mask_bits);
        const int cols = min(kTile, T2 - c0);
        float* blk = a.out + (static_cast<size_t>(bh) * T + r0) * T2 + c0;
        for (int rr = 0; rr < kTile && r0 + rr < T; ++rr)
          for (int i = static_cast<int>(lane); i < cols; i += 32)
            blk[static_cast<size_t>(rr) * T2 + i] = m;
      }
    }
    // Only the stores' reads of shared memory must finish before the CTA exits;
    // their global writes complete before the grid does.
    if (lane == 0) bulk_wait_read<0>();
    __syncwarp();
  } else {
    // ---------------------------------------------------------- epilogue --
    // Warp e = warp - 2 owns the 32 rows of TMEM lane quarter warp % 4 (a warp may
    // only read the lanes of its quarter) and the 64-column slab e / 4 of the tile:
    // one 64-column TMEM load, one proxy fence and one commit group per tile.
    const uint32_t ew = warp - 2u;
    const int q = static_cast<int>(warp & 3u);
    const int slab = static_cast<int>(ew >> 2);
    const uint32_t staging = base + a.off_staging + ew * a.staging_stride;
    const int T = a.T, T2 = a.T2;  // output rows and columns of one (b, h)
    int acc = 0;
    uint32_t acc_phase = 0;
    uint32_t grp = 0;
    int slot = 0;
    uint32_t sphase = 0;
    while (true) {
      int ok = 1;
      unsigned int cur = 0;
      if (lane == 0) {
        ok = mbar_wait(sfull_bar(slot), sphase, wd, kSiteSched) ? 1 : 0;
        if (ok) {
          cur = ld_shared_b32(sched_entry(slot));
          mbar_arrive(sempty_bar(slot));
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      cur = __shfl_sync(0xffffffffu, cur, 0);
      if (!ok || cur == kEntryEnd) break;
      if (++slot == kSchedDepth) {
        slot = 0;
        sphase ^= 1u;
      }
      int bh, rank, ti, tj;
      decode_position(static_cast<int>(cur), a.per_lower, bh, rank);
      decode_computed(rank, a.causal, a.Tt2, ti, tj);
      if (!CSA_CHECK(bh >= 0 && bh < a.BH && ti >= 0 && ti < a.Tt && tj >= 0 && tj < a.Tt2 &&
                         acc * kTile + (slab + 1) * kSlabCols <= static_cast<int>(a.tmem_cols),
                     wd, kCheckTile))
        break;
      const int row0 = ti * kTile + q * 32;
      const int colw = tj * kTile + slab * kSlabCols;

      // Idle while the accumulator is not ready: the fill writer may store then.
      if (ew == 0 && lane == 0) *epi_idle = 1;
      const bool got = mbar_wait_warp(tfull_bar(acc), acc_phase, wd, kSiteEpilogueFull);
      if (ew == 0 && lane == 0) *epi_idle = 0;
      if (!got) break;
      tc_fence_after_sync();
      uint32_t v[kSlabCols];
      tmem_ld_64cols(tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                         static_cast<uint32_t>(acc * kTile + slab * kSlabCols),
                     v);
      // This warp's part of the accumulator is in registers: release it.
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty_bar(acc));
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }

      const bool diag = a.causal && ti == tj;
      const int r = row0 + static_cast<int>(lane);
      if (!diag) {
#pragma unroll
        for (int e = 0; e < kSlabCols; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * a.scale);
      } else {
#pragma unroll
        for (int e = 0; e < kSlabCols; ++e)
          v[e] = (colw + e > r) ? a.mask_bits : __float_as_uint(__uint_as_float(v[e]) * a.scale);
      }
      if (row0 >= T || colw >= T2) continue;  // slab wholly past the end (tail tile)

      // Per 32-column box: 0 skip, 1 TMA store, 2 plain stores, 3 plain stores t2 <= t
      // only, 4 (16-byte-aligned rows) each lane stores its row's t2 <= t part from
      // registers with vector stores.
      int mode[2];
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int col0 = colw + c * 32;
        mode[c] = col0 >= T2 ? 0 : (a.tma_store ? 1 : 2);
        if (mode[c] != 0 && a.lower_only && diag) {
          if (col0 > row0 + 31) mode[c] = 0;
          else if (col0 + 31 > row0) mode[c] = a.tma_store ? 4 : 3;
        }
      }
      if (mode[0] == 0 && mode[1] == 0) continue;

      if constexpr (kSingleBox) {
        {
          // One staging box per warp (more room for the operand rings): the two
          // 32-column boxes go out one after the other.
          for (int c = 0; c < 2; ++c) {
            if (mode[c] == 0) continue;
            if (lane == 0) bulk_wait_read<0>();
            __syncwarp();
            stage_row_sw128(staging, lane, v + 32 * c);
            if (mode[c] == 1) {
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                tma_store_3d(&tmap_out, staging, colw + c * 32, row0, bh);
                bulk_commit();
              }
              continue;
            }
            __syncwarp();
            const int col = colw + c * 32 + static_cast<int>(lane);
            float* ocol = a.out + (static_cast<size_t>(bh) * T + row0) * T2 + col;
            for (int rr = 0; rr < 32; ++rr) {
              const int row = row0 + rr;
              const bool ok = row < T && col < T2 && (mode[c] == 2 || col <= row);
              const uint32_t val = staged_elem_sw128(staging, static_cast<uint32_t>(rr), lane);
              if (ok) ocol[static_cast<size_t>(rr) * T2] = __uint_as_float(val);
            }
            __syncwarp();
          }
          continue;
        }
      }

      if (lane == 0) {
        if (a.store_groups == 2) bulk_wait_read<1>();
        else bulk_wait_read<0>();
      }
      __syncwarp();
      const uint32_t pair = staging + grp * 2u * kBoxBytes;
      if (++grp == a.store_groups) grp = 0;
#pragma unroll
      for (int c = 0; c < 2; ++c)
        if (mode[c] != 0 && mode[c] != 4) stage_row_sw128(pair + c * kBoxBytes, lane, v + 32 * c);
      const bool any_tma = mode[0] == 1 || mode[1] == 1;
      if (any_tma) fence_proxy_async_smem();
      __syncwarp();
      if (any_tma && lane == 0) {
        for (int c = 0; c < 2; ++c)
          if (mode[c] == 1) tma_store_3d(&tmap_out, pair + c * kBoxBytes, colw + c * 32, row0, bh);
        bulk_commit();
      }
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        if (mode[c] != 4 || r >= T) continue;
        const int c0 = colw + c * 32;
        const int lim = r - c0;  // this row's columns c0 + e, e <= lim, are t2 <= t
        float* orow = a.out + (static_cast<size_t>(bh) * T + r) * T2 + c0;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int e0 = 4 * k;
          if (e0 + 3 <= lim) {
            *reinterpret_cast<float4*>(orow + e0) =
                make_float4(__uint_as_float(v[32 * c + e0]), __uint_as_float(v[32 * c + e0 + 1]),
                            __uint_as_float(v[32 * c + e0 + 2]), __uint_as_float(v[32 * c + e0 + 3]));
          } else {
#pragma unroll
            for (int j = 0; j < 4; ++j)
              if (e0 + j <= lim) orow[e0 + j] = __uint_as_float(v[32 * c + e0 + j]);
          }
        }
      }
      for (int c = 0; c < 2; ++c) {
        if (mode[c] < 2 || mode[c] == 4) continue;
        const int col = colw + c * 32 + static_cast<int>(lane);
        float* ocol = a.out + (static_cast<size_t>(bh) * T + row0) * T2 + col;
        for (int rr = 0; rr < 32; ++rr) {
          const int row = row0 + rr;
          const bool ok = row < T && col < T2 && (mode[c] == 2 || col <= row);
          const uint32_t val =
              staged_elem_sw128(pair + c * kBoxBytes, static_cast<uint32_t>(rr), lane);
          if (ok) ocol[static_cast<size_t>(rr) * T2] = __uint_as_float(val);
        }
      }
    }
    if (ew == 0 && lane == 0) *epi_idle = 1;
    // Only the stores' reads of shared memory must finish before the CTA exits;
    // their global writes complete before the grid does.
    if (lane == 0) bulk_wait_read<0>();
    __syncwarp();
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, static_cast<uint32_t>(a.tmem_cols));
  }
  if (threadIdx.x == 0 && (a.dynamic || a.n_fill > 0)) {
    // Every fetch of this CTA is done; the last CTA to get here resets the pair.
    // (A static deal without fill tiles never touches the counters: no reset, and
    // no fence and atomics on every CTA's way out.)
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

namespace {

// One launch of the score kernel over BH (b, h) problems with T x T2 outputs
// each, given the operand tensor maps (A rows index t, B rows index t2).
int launch_scores(const char* who, const CUtensorMap& map_a, const CUtensorMap& map_b, float* out,
                  long long BH, int T, int T2, int D, int nh_div, int b_off, bool causal,
                  bool lower_only, float scale, uint32_t mask_bits, bool inject,
                  cudaStream_t stream, const DeviceInfo& dev, std::string& err,
                  unsigned int* counters, bool f32 = false) {
  const std::string name(who);
  if (BH > (1LL << 30) || static_cast<long long>(T) > (1LL << 30) ||
      static_cast<long long>(T2) > (1LL << 30)) {
    err = name + ": too many (b, h) problems or too long a sequence";
    return CSA_ERR_SHAPE;
  }
  TrimulArgs a{};
  a.T = T;
  a.T2 = T2;
  a.BH = static_cast<int>(BH);
  a.Tt = (T + kTile - 1) / kTile;
  a.Tt2 = (T2 + kTile - 1) / kTile;
  a.nh_div = nh_div;
  a.b_off = b_off;
  a.causal = causal ? 1u : 0u;
  // bf16: a stage holds all of a tile's 64-element chunks. fp32 (3xtf32): a
  // stage holds one 32-element chunk of Q and K plus their lo parts.
  a.chunk_elems = f32 ? kChunkElemsF32 : kChunkElems;
  a.kchunks = (D + a.chunk_elems - 1) / a.chunk_elems;
  a.ksteps = (D + 15) / 16;
  a.stage_chunks = f32 ? 1 : a.kchunks;
  a.tile_stages = f32 ? a.kchunks : 1;
  const long long per_lower = causal ? static_cast<long long>(a.Tt) * (a.Tt + 1) / 2
                                     : static_cast<long long>(a.Tt) * a.Tt2;
  const long long per_fill =
      (causal && !lower_only) ? static_cast<long long>(a.Tt) * (a.Tt - 1) / 2 : 0;
  if (BH * per_lower >= (1LL << 31) - (1LL << 20) || BH * per_fill >= (1LL << 31) - (1LL << 20) ||
      per_lower + per_fill >= (1LL << 20)) {
    err = name + ": too many tiles";
    return CSA_ERR_SHAPE;
  }
  a.n_lower = static_cast<int>(BH * per_lower);
  a.n_fill = static_cast<int>(BH * per_fill);
  a.per_lower = static_cast<int>(per_lower);
  a.per_fill = static_cast<int>(per_fill);
  // fp32 with HS <= 128: Q's hi / lo parts (2 x 32 columns per chunk) fit in
  // TMEM beside the two accumulators; CTAs then take contiguous runs of tiles.
  const bool q_tmem = f32 && a.kchunks <= (512 - kTmemCols) / 64;
  a.q_tmem = q_tmem ? 1u : 0u;
  a.contig = q_tmem ? 1u : 0u;
  a.tmem_cols = q_tmem ? 512 : kTmemCols;
  // Two Q buffers when both fit beside the accumulators (2 x 64 columns per chunk).
  a.q_bufs = (q_tmem && CSA_TRIMUL_Q_BUFS > 1 && kTmemCols + 2 * 64 * a.kchunks <= 512) ? 2 : 1;
  a.dynamic = (!q_tmem && a.n_fill > 0) ? 1u : 0u;
  a.scale = scale;
  a.mask_bits = mask_bits;
  a.lower_only = lower_only ? 1u : 0u;
  a.tma_store = (T2 % 4 == 0 && reinterpret_cast<uintptr_t>(out) % 16 == 0) ? 1u : 0u;
  a.out = out;
  a.status = dev.status_word;
  a.wait_limit_ns = wait_limit_ns();
  a.inject = inject ? 1 : 0;

  // Shared memory: operand ring | staging boxes | mask buffer | barriers | misc.
  // Operand ring stages vs. staging depth: the most box pairs per epilogue warp
  // that still leave two ring stages, else one pair.
  a.stage_bytes = f32 ? (q_tmem ? 1u : 4u) * kChunkBytes
                      : static_cast<uint32_t>(a.kchunks) * 2u * kChunkBytes;
  a.lo_slots = q_tmem ? CSA_TRIMUL_LO_SLOTS : 0;
  const int lo_bytes = a.lo_slots * kChunkBytes;
  // The mask buffer only exists when there are fill tiles (full causal mode).
  const int fill_bytes = a.n_fill > 0 ? kFillBytes : 0;
  const int fixed = fill_bytes + lo_bytes + 1024 /*bars+misc+ring*/ + 1024 /*align slack*/;
  const int max_stages = q_tmem ? CSA_TRIMUL_MAX_STAGES_QT : CSA_TRIMUL_MAX_STAGES;
  int staging_bytes = 0;
  for (int groups = CSA_TRIMUL_MAX_STORE_GROUPS; groups >= 1; --groups) {
    staging_bytes = kEpiWarps * groups * 2 * kBoxBytes;
    a.store_groups = static_cast<uint32_t>(groups);
    a.stages = std::min(max_stages, (dev.max_smem_optin - fixed - staging_bytes) /
                                        static_cast<int>(a.stage_bytes));
    if (a.stages >= 2) break;
  }
  const bool single_box = q_tmem && CSA_TRIMUL_F32_SINGLE_BOX && a.n_fill > 0;
  if (single_box) {
    // fp32 with Q in TMEM: one staging box per epilogue warp (store_groups 0); its
    // epilogue mostly waits on the MMAs, and the operand rings take the space.
    staging_bytes = kEpiWarps * kBoxBytes;
    a.store_groups = 0u;
    a.stages = std::min(max_stages, (dev.max_smem_optin - fixed - staging_bytes) /
                                        static_cast<int>(a.stage_bytes));
  }
  a.staging_stride = static_cast<uint32_t>(staging_bytes / kEpiWarps);
  if (a.stages < 1) {
    err = name + ": not enough shared memory for one operand stage";
    return CSA_ERR_UNSUPPORTED;
  }
  a.off_lo = static_cast<uint32_t>(a.stages) * a.stage_bytes;
  a.off_staging = a.off_lo + static_cast<uint32_t>(lo_bytes);
  a.off_mask = a.off_staging + static_cast<uint32_t>(staging_bytes);
  a.off_bars = a.off_mask + static_cast<uint32_t>(fill_bytes);
  a.off_misc =
      a.off_bars + 8u * static_cast<uint32_t>(3 * a.stages + 7 + 2 * kSchedDepth + a.lo_slots);
  const size_t smem = a.off_misc + 16 + 4 * kSchedDepth + 1024;

  CUtensorMap map_out, map_fill;
  if (a.tma_store) {
    const uint64_t dims[3] = {static_cast<uint64_t>(T2), static_cast<uint64_t>(T),
                              static_cast<uint64_t>(BH)};
    const uint64_t strides[2] = {static_cast<uint64_t>(T2) * 4,
                                 static_cast<uint64_t>(T) * static_cast<uint64_t>(T2) * 4};
    const uint32_t box[3] = {32, 32, 1};
    int rc = encode_tiled(&map_out, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, out, dims, strides, box,
                          CU_TENSOR_MAP_SWIZZLE_128B, err);
    if (rc != CSA_OK) return rc;
    const uint32_t fbox[3] = {kFillCols, kFillRows, 1};
    rc = encode_tiled(&map_fill, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, out, dims, strides, fbox,
                      CU_TENSOR_MAP_SWIZZLE_NONE, err);
    if (rc != CSA_OK) return rc;
  } else {
    std::memset(&map_out, 0, sizeof map_out);
    std::memset(&map_fill, 0, sizeof map_fill);
  }

  CounterSlot slot;
  if (counters) {
    a.sched = counters;  // caller-provided counters (zeroed before this launch)
  } else if (a.dynamic || a.n_fill > 0) {
    static std::mutex mu;
    static unsigned int* sched_base[64] = {};
    {
      std::lock_guard<std::mutex> lock(mu);
      if (dev.device < 0 || dev.device >= 64) {
        err = name + ": device ordinal out of range";
        return CSA_ERR_CUDA;
      }
      if (!sched_base[dev.device]) {
        void* p = nullptr;
        cudaError_t se = cudaGetSymbolAddress(&p, g_trimul_sched);
        if (se != cudaSuccess) {
          err = name + ": cudaGetSymbolAddress: " + cudaGetErrorString(se);
          return CSA_ERR_CUDA;
        }
        sched_base[dev.device] = static_cast<unsigned int*>(p);
      }
    }
    int rc = acquire_counter_slot(kFamilyScores, dev, sched_base[dev.device], stream, slot, err);
    if (rc != CSA_OK) {
      err = name + ": " + err;
      return rc;
    }
    a.sched = slot.counters;
    a.done = slot.done;
    a.seq = slot.seq;
  }
  // (a static deal without fill tiles never touches the counters: no set at all)
  auto* kernel = !f32         ? trimul_sm103a_kernel<false, false>
                 : single_box ? trimul_sm103a_kernel<true, true>
                              : trimul_sm103a_kernel<true, false>;
  {
    int rc = set_max_dynamic_smem(reinterpret_cast<const void*>(kernel), static_cast<int>(smem),
                                  dev.device, err);
    if (rc != CSA_OK) {
      abandon_counter_slot(kFamilyScores, dev, slot);
      err = name + ": " + err;
      return rc;
    }
  }
  cudaError_t e;
  const long long grid = std::min<long long>(static_cast<long long>(a.n_lower) + a.n_fill,
                                            dev.sm_count);
  e = launch_programmatic(kernel, static_cast<unsigned>(grid), f32 ? kThreadsF32 : kThreads, smem,
                          stream, map_a, map_b, map_out, map_fill, a);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) {
    abandon_counter_slot(kFamilyScores, dev, slot);
    err = name + ": launch: " + cudaGetErrorString(e);
    return CSA_ERR_LAUNCH;
  }
  return CSA_OK;
}

}  // namespace

int trimul_launch(float* out, const void* qkv, int B, int T, int C, int NH, uint32_t mask_bits,
                  uint32_t flags, cudaStream_t stream, const DeviceInfo& dev, std::string& err,
                  unsigned int* counters) {
  const int HS = C / NH;
  if (HS % 8 != 0) {
    err = "trimul_forward: HS = C/NH must be a multiple of 8 (TMA row pitch of a head)";
    return CSA_ERR_ALIGN;
  }
  if (HS > 256) {
    err = "trimul_forward: HS > 256 is not supported";
    return CSA_ERR_UNSUPPORTED;
  }
  if (reinterpret_cast<uintptr_t>(qkv) % 16 != 0 || reinterpret_cast<uintptr_t>(out) % 4 != 0) {
    err = "trimul_forward: qkv must be 16-byte aligned and out 4-byte aligned";
    return CSA_ERR_ALIGN;
  }
  // Q of head h is index h and its key index NH + h along the (3, NH) axis of
  // the packed tensor, read in place.
  CUtensorMap map_qkv;
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
  const float scale = static_cast<float>(1.0 / std::sqrt(static_cast<double>(HS)));
  return launch_scores("trimul_forward", map_qkv, map_qkv, out, static_cast<long long>(B) * NH, T,
                       T, HS, NH, NH, true, (flags & CSA_TRIMUL_LOWER_ONLY) != 0, scale,
                       mask_bits, take_inject(), stream, dev, err, counters);
}

int trimul_f32_launch(float* out, const float* qkv, int B, int T, int C, int NH,
                      uint32_t mask_bits, uint32_t flags, cudaStream_t stream, const DeviceInfo& dev,
                      std::string& err) {
  const int HS = C / NH;
  if (HS % 4 != 0) {
    err = "trimul_forward_f32: HS = C/NH must be a multiple of 4 (TMA row pitch of a head)";
    return CSA_ERR_ALIGN;
  }
  if (HS > 256) {
    err = "trimul_forward_f32: HS > 256 is not supported";
    return CSA_ERR_UNSUPPORTED;
  }
  if (reinterpret_cast<uintptr_t>(qkv) % 16 != 0 || reinterpret_cast<uintptr_t>(out) % 4 != 0) {
    err = "trimul_forward_f32: qkv must be 16-byte aligned and out 4-byte aligned";
    return CSA_ERR_ALIGN;
  }
  // The packed fp32 tensor read in place: Q of head h at index h, K at NH + h.
  CUtensorMap map_qkv;
  {
    const uint64_t dims[4] = {static_cast<uint64_t>(HS), static_cast<uint64_t>(3 * NH),
                              static_cast<uint64_t>(T), static_cast<uint64_t>(B)};
    const uint64_t strides[3] = {static_cast<uint64_t>(HS) * 4, static_cast<uint64_t>(C) * 12,
                                 static_cast<uint64_t>(T) * C * 12};
    const uint32_t box[4] = {kChunkElemsF32, 1, kTile, 1};
    int rc = encode_tiled(&map_qkv, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, qkv, dims, strides, box,
                          CU_TENSOR_MAP_SWIZZLE_128B, err);
    if (rc != CSA_OK) return rc;
  }
  const float scale = static_cast<float>(1.0 / std::sqrt(static_cast<double>(HS)));
  return launch_scores("trimul_forward_f32", map_qkv, map_qkv, out, static_cast<long long>(B) * NH,
                       T, T, HS, NH, NH, true, (flags & CSA_TRIMUL_LOWER_ONLY) != 0, scale,
                       mask_bits, take_inject(), stream, dev, err, nullptr, true);
}

int bmm_nt_launch(float* Y, const void* X, const void* W, int batch, int T1, int T2, int D,
                  cudaStream_t stream, const DeviceInfo& dev, std::string& err) {
  if (D % 8 != 0) {
    err = "batch_matmul_nt: D must be a multiple of 8 (TMA row pitch)";
    return CSA_ERR_ALIGN;
  }
  if (D > 256) {
    err = "batch_matmul_nt: D > 256 is not supported";
    return CSA_ERR_UNSUPPORTED;
  }
  if (reinterpret_cast<uintptr_t>(X) % 16 != 0 || reinterpret_cast<uintptr_t>(W) % 16 != 0 ||
      reinterpret_cast<uintptr_t>(Y) % 4 != 0) {
    err = "batch_matmul_nt: X and W must be 16-byte aligned and Y 4-byte aligned";
    return CSA_ERR_ALIGN;
  }
  // X [batch, T1, D] and W [batch, T2, D] as 4-D maps (D, 1, rows, batch) so the
  // kernel addresses them like the packed tensor with a single head.
  CUtensorMap map_x, map_w;
  for (int which = 0; which < 2; ++which) {
    const int rows = which == 0 ? T1 : T2;
    const uint64_t dims[4] = {static_cast<uint64_t>(D), 1, static_cast<uint64_t>(rows),
                              static_cast<uint64_t>(batch)};
    const uint64_t strides[3] = {static_cast<uint64_t>(D) * 2, static_cast<uint64_t>(D) * 2,
                                 static_cast<uint64_t>(rows) * D * 2};
    const uint32_t box[4] = {kChunkElems, 1, kTile, 1};
    int rc = encode_tiled(which == 0 ? &map_x : &map_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
                          which == 0 ? X : W, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B, err);
    if (rc != CSA_OK) return rc;
  }
  return launch_scores("batch_matmul_nt", map_x, map_w, Y, batch, T1, T2, D, 1, 0, false, false,
                       1.0f, 0u, false, stream, dev, err, nullptr);
}

// ---------------------------------------------------- allocation-free variant --
//
// Scratch of trimul_launch_noalloc: the work-list counter pair the kernel needs,
// in a fixed array that every device loading this library holds until exit
// (no cudaMalloc anywhere on that path). One array per device, shared by every
// call on that device, so calls whose kernels overlap on the GPU race on it.
constexpr size_t kNoallocScratchBytes = 256;
static __device__ __align__(256) unsigned int g_trimul_noalloc_scratch[kNoallocScratchBytes / 4];

int trimul_launch_noalloc(float* out, const void* qkv, int B, int T, int C, int NH,
                          uint32_t mask_bits, uint32_t flags, cudaStream_t stream,
                          const DeviceInfo& dev, std::string& err) {
  // What this call keeps in the scratch: the kernel's 32-bit work-list counters.
  constexpr size_t kNeeded = kSchedWords * sizeof(unsigned int);
  static_assert(kNeeded <= kNoallocScratchBytes, "scratch array too small");
  // The counters index the work list; a list beyond their range is rejected.
  const long long Tt = (static_cast<long long>(T) + kTile - 1) / kTile;
  const long long tiles = static_cast<long long>(B) * NH * Tt * Tt;
  if (tiles >= (1LL << 31) - (1LL << 20)) {
    err = "trimul_forward_noalloc: " + std::to_string(tiles) +
          " output tiles exceed what its fixed scratch counters can index (2^31 - 2^20)";
    return CSA_ERR_SHAPE;
  }
  // Set-up, once per device, with that device current: the device address of the
  // scratch array (its name is only a host-side stand-in in host code).
  static std::mutex mu;
  static unsigned int* scratch[64] = {};
  unsigned int* counters = nullptr;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (dev.device < 0 || dev.device >= 64) {
      err = "trimul_forward_noalloc: device ordinal out of range";
      return CSA_ERR_CUDA;
    }
    if (!scratch[dev.device]) {
      void* p = nullptr;
      const cudaError_t e = cudaGetSymbolAddress(&p, g_trimul_noalloc_scratch);
      if (e != cudaSuccess || !p) {
        err = std::string("trimul_forward_noalloc: cudaGetSymbolAddress: ") +
              cudaGetErrorString(e);
        return CSA_ERR_CUDA;
      }
      scratch[dev.device] = static_cast<unsigned int*>(p);
    }
    counters = scratch[dev.device];
  }
  // The counters must start at zero; the array keeps whatever the last call left.
  const cudaError_t e = cudaMemsetAsync(counters, 0, kNeeded, stream);
  if (e != cudaSuccess) {
    err = std::string("trimul_forward_noalloc: clearing scratch: ") + cudaGetErrorString(e);
    return CSA_ERR_CUDA;
  }
  return trimul_launch(out, qkv, B, T, C, NH, mask_bits, flags, stream, dev, err, counters);
}

}  // namespace csa

#ifdef CSA_DEBUG
// Checking build only: fills the allocation-free entry point's scratch with
// `value` in every word, as an earlier launch that stopped mid-list would leave
// its counters, so that a test can see each call clear them before its kernel.
extern "C" csa_status csa_debug_noalloc_scratch_fill(uint32_t value) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, csa::g_trimul_noalloc_scratch) != cudaSuccess) return CSA_ERR_CUDA;
  uint32_t words[csa::kNoallocScratchBytes / 4];
  for (uint32_t& w : words) w = value;
  return cudaMemcpy(p, words, sizeof words, cudaMemcpyHostToDevice) == cudaSuccess ? CSA_OK
                                                                                   : CSA_ERR_CUDA;
}
#endif
