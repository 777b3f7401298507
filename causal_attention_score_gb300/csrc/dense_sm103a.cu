// Ragged dense layer on sm_103a: Y[M, H] = X[M, I] W[H, I]^T, bf16 in, fp32 out.
//
// The workload is the dense layer of "DietCode tests/codegen/
// test_1_local_padding.py" (test_local_padding docstring), whose point is
// "local padding": the bounds checks of an imperfectly tiled product belong
// only to the Fetch stage (out-of-range elements become zeros) and the
// Writeback stage (out-of-range results are not stored); the Compute stage
// then runs over whole tiles with no predicates at all.
//
// Design (one persistent launch, one CTA per SM, 9 warps):
//  - tiles of 128 x BN outputs (BN = 64, 128, 192 or 256, chosen per shape),
//    K in blocks of 64; tiles are dealt round-robin to CTAs.
//  - dense_xwt_grouped: up to 48 problems sharing W in one launch (their tensor
//    maps in the kernel parameters, m-tiles of all problems in one list); when
//    the occupancy allows it, clusters of two CTAs compute 256 x BN tiles as a
//    CTA pair (tcgen05 cta_group::2), each CTA holding 128 rows.
//  - Fetch, two forms:
//      * TMA (I*2 % 16 == 0, 16-byte aligned X and W): warp 0 issues 2-D tiled
//        loads; rows >= M / H and columns >= I are zero-filled by the TMA unit.
//        Rows that no tensor map can describe (e.g. I = 770: 1540-byte rows)
//        are first copied by realign_rows_kernel into the caller's workspace
//        as rows that start on 128-byte boundaries (pitch I rounded up to 64
//        elements); the tiles are then fetched from that copy by TMA, with the
//        same zero fill at the edges. The copy only moves rows: no padding to
//        tile multiples is materialised.
//      * loader warps (rows no tensor map can describe, with no workspace):
//        warps 0-3 read 4-byte (or 2-byte) pairs with plain loads, substitute
//        zeros out of range, and write them into the same 128-byte-swizzled
//        K-major layout the TMA would produce.
//  - Compute: warp 4 issues tcgen05.mma M=128 N=BN K=16 into one of two TMEM
//    accumulators; no bounds logic at all.
//  - Writeback: warps 5-8 read TMEM 32 columns at a time and store 32 x 32
//    boxes with TMA (clipped at M and H) when Y rows are 16-byte aligned, or
//    with coalesced predicated plain stores otherwise.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <string>

#include "csa_internal.h"
#include "sm103a_ptx.cuh"

namespace csa {
namespace {

constexpr int kBM = 128;
constexpr int kBK = 64;
constexpr int kThreads = 288;
constexpr int kLoaderWarps = 4;
constexpr int kMmaWarp = 4;
constexpr int kFirstEpiWarp = 5;
#ifndef CSA_DENSE_MAX_STAGES
#define CSA_DENSE_MAX_STAGES 8
#endif
// Groups: clusters of two CTAs computing 256-row tiles as a CTA pair (1), or one
// CTA per 128-row tile (0).
#ifndef CSA_DENSE_PAIR
#define CSA_DENSE_PAIR 1
#endif
// One problem (dense_xwt): CTA pairs when the tiling model prefers them (-1),
// never (0), always when the rows are fetched by TMA (1).
#ifndef CSA_DENSE_SINGLE_PAIR
#define CSA_DENSE_SINGLE_PAIR -1
#endif
#ifndef CSA_DENSE_STORE_BUFS
#define CSA_DENSE_STORE_BUFS 2
#endif
constexpr int kStoreBufs = CSA_DENSE_STORE_BUFS;  // staging boxes per epilogue warp
constexpr int kBoxBytes = 32 * 32 * 4;
constexpr int kStagingBytes = 4 * kStoreBufs * kBoxBytes;

struct DenseArgs {
  int M, I, H, BN;
  int m_tiles, n_tiles, kblocks, stages;
  long long num_tiles;
  uint32_t tma_load, tma_store, vec2;
  int load_depth;  // cp.async stages in flight per loader warp (2..4, <= stages)
  int inject;      // withhold each CTA's first operand hand-off (watchdog tests)
  uint32_t idesc;
  const uint16_t* X;
  const uint16_t* W;
  float* Y;
  int* status;
  unsigned long long wait_limit_ns;
  uint32_t stage_bytes, off_staging, off_bars, off_misc, tmem_cols;
};

// Grouped launch: up to kMaxGroup problems Y[g] = X[g] W^T that share W, I and
// H, one persistent launch over all their tiles. The per-problem tensor maps
// travel in the kernel parameters (nothing to allocate, so a grouped call can be
// captured in a CUDA graph).
constexpr int kMaxGroup = 48;
template <bool kGrouped>
struct DenseGroup {};  // one problem: everything is in DenseArgs and the three maps
template <>
struct DenseGroup<true> {
  CUtensorMap x[kMaxGroup];     // X[g] as (I, M[g]), 64 x 128 boxes
  CUtensorMap y[kMaxGroup];     // Y[g] as (H, M[g]), 32 x 32 boxes (TMA store form)
  float* Y[kMaxGroup];
  int M[kMaxGroup];
  int mt_start[kMaxGroup + 1];  // first m-tile of problem g in the launch; [n] = all
  int n;
};

template <bool kPair>
__device__ __forceinline__ uint32_t load_pair(const uint16_t* row, int k, int I) {
  if (kPair) {
    // I even and 4-byte aligned rows: k is even, so k < I covers both halves.
    return k < I ? __ldg(reinterpret_cast<const unsigned int*>(row + k)) : 0u;
  } else {
    const uint32_t lo = k < I ? __ldg(reinterpret_cast<const unsigned short*>(row + k)) : 0u;
    const uint32_t hi = k + 1 < I ? __ldg(reinterpret_cast<const unsigned short*>(row + k + 1)) : 0u;
    return lo | (hi << 16);
  }
}

__device__ __forceinline__ uint32_t swz_row_word(uint32_t tile, uint32_t rl, uint32_t lane) {
  // bf16 pair (2*lane, 2*lane+1) of row rl in the 128-byte-swizzle K-major layout
  return tile + rl * 128u + ((((lane >> 2) ^ (rl & 7u))) << 4) + ((lane & 3u) << 2);
}

// One loader warp's share of a rows x 64 operand block: rows w, w+4, w+8, ...
// Each lane handles bf16 columns k, k+1 (k = kb*64 + 2*lane); the warp writes
// whole 128-byte rows, so the swizzled stores are bank-conflict free.
// Synchronous form (plain loads into registers, then st.shared), used for odd I.
template <bool kPair>
__device__ __forceinline__ void load_block(const uint16_t* src, int nrows, int row_base, int rows,
                                           int I, int k, uint32_t tile, uint32_t w,
                                           uint32_t lane) {
  for (int i0 = 0; i0 < rows / kLoaderWarps; i0 += 8) {
    uint32_t v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int rl = (i0 + u) * kLoaderWarps + static_cast<int>(w);
      const int row = row_base + rl;
      v[u] = row < nrows ? load_pair<kPair>(src + static_cast<size_t>(row) * I, k, I) : 0u;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const uint32_t rl = static_cast<uint32_t>((i0 + u) * kLoaderWarps) + w;
      st_shared_b32(swz_row_word(tile, rl, lane), v[u]);
    }
  }
}

// Asynchronous form (I even, 4-byte aligned rows): one 4-byte cp.async per lane
// and row; out-of-range pairs are zero-filled by a source size of 0.
__device__ __forceinline__ void issue_block_async(const uint16_t* src, int nrows, int row_base,
                                                  int rows, int I, int k, uint32_t tile,
                                                  uint32_t w, uint32_t lane) {
  const bool k_in = k < I;
  for (int i = 0; i < rows / kLoaderWarps; ++i) {
    const uint32_t rl = static_cast<uint32_t>(i * kLoaderWarps) + w;
    const int row = row_base + static_cast<int>(rl);
    const bool in = k_in && row < nrows;
    const uint16_t* p = in ? src + static_cast<size_t>(row) * I + k : src;
    cp_async_4(swz_row_word(tile, rl, lane), p, in ? 4u : 0u);
  }
}

// kPair: clusters of two CTAs compute 256-row tiles as a CTA pair
// (tcgen05 cta_group::2): each CTA loads its own 128 rows of X and half of the W
// tile's rows, and the pair's first CTA issues M = 256 MMAs that read both CTAs'
// shared memory, each CTA's TMEM receiving its own rows. Per k-block each SM then
// receives (128 + BN/2) x 128 bytes instead of (128 + BN) x 128. Both CTAs' loads
// complete on the first CTA's full barrier; its commits go to both CTAs' barriers;
// the second CTA's epilogue releases accumulators on the first CTA's barrier.
template <bool kGrouped, bool kPair = false>
__global__ void __launch_bounds__(kThreads, 1)
    dense_sm103a_kernel(const __grid_constant__ CUtensorMap tmap_x,
                        const __grid_constant__ CUtensorMap tmap_w,
                        const __grid_constant__ CUtensorMap tmap_y, const DenseArgs a,
                        const __grid_constant__ DenseGroup<kGrouped> g) {
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
  const uint32_t tmem_slot = base + a.off_misc;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + a.off_misc + 4);
  auto a_tile = [&](int s) { return base + s * a.stage_bytes; };
  auto b_tile = [&](int s) { return base + s * a.stage_bytes + kBM * 128u; };

  const Watchdog wd{a.wait_limit_ns, a.status, abort_flag};

  // With kPair, this CTA's half of each tile pair (0 or 1) and the pair walk.
  const uint32_t rank = kPair ? cluster_ctarank() : 0u;
  const long long t_first = kPair ? blockIdx.x / 2 : blockIdx.x;
  const long long t_step = kPair ? gridDim.x / 2 : gridDim.x;

  // Tile t of the launch: problem p, its m-tile mb, the n-tile nb. A group is
  // m-major (the n-tiles of one m-tile follow one another, so CTAs working at the
  // same time share X's m-tile and spread their reads over all of W; n-major, every
  // CTA read the same W tile at once: measured 8 % slower on the grouped sweep),
  // the m-tiles of all problems following one another. One problem is n-major
  // (measured 2 % faster than m-major over the sweep's separate calls).
  auto locate = [&](long long t, int& p, int& mb, int& nb) {
    if constexpr (!kGrouped && kPair) {
      // One problem in pairs: t numbers (pair of m-tiles, n-tile), n-major; the
      // phantom half of a pair past the last m-tile is zero-filled and not stored.
      const long long m_pairs = (a.m_tiles + 1) / 2;
      p = 0;
      mb = static_cast<int>(2 * (t % m_pairs) + rank);
      nb = static_cast<int>(t / m_pairs);
    } else if constexpr (kGrouped) {
      // (pairs: t numbers tile pairs; a pair past the last m-tile has a phantom
      // half, whose rows are past its problem's M: zero-filled and not stored)
      const int mt = kPair ? static_cast<int>(2 * (t / a.n_tiles) + rank)
                           : static_cast<int>(t / a.n_tiles);
      nb = static_cast<int>(t % a.n_tiles);
      int lo = 0, hi = g.n - 1;  // the last problem whose first m-tile is <= mt
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (g.mt_start[mid] <= mt) lo = mid;
        else hi = mid - 1;
      }
      p = lo;
      mb = mt - g.mt_start[lo];
    } else {
      p = 0;
      mb = static_cast<int>(t % a.m_tiles);
      nb = static_cast<int>(t / a.m_tiles);
    }
  };
#ifdef CSA_DEBUG
  // A located tile lies inside the launch's problems and n-tiles (with kPair the
  // phantom half past the last m-tile is allowed).
  auto tile_ok = [&](int p, int mb, int nb) {
    int n = 1;
    if constexpr (kGrouped) n = g.n;
    return p >= 0 && p < n && mb >= 0 && nb >= 0 && nb < a.n_tiles &&
           (kGrouped || mb < a.m_tiles + (kPair ? 1 : 0));
  };
#endif
  auto map_x = [&](int p) -> const CUtensorMap* {
    if constexpr (kGrouped) return &g.x[p];
    else return &tmap_x;
  };
  auto map_y = [&](int p) -> const CUtensorMap* {
    if constexpr (kGrouped) return &g.y[p];
    else return &tmap_y;
  };
  auto rows_of = [&](int p) -> int {
    if constexpr (kGrouped) return g.M[p];
    else return a.M;
  };
  auto y_of = [&](int p) -> float* {
    if constexpr (kGrouped) return g.Y[p];
    else return a.Y;
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < a.stages; ++s) {
      mbar_init(full_bar(s), a.tma_load ? 1u : static_cast<uint32_t>(kLoaderWarps));
      mbar_init(empty_bar(s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(tfull_bar(s), 1);
      mbar_init(tempty_bar(s), kPair ? 8u : 4u);  // with kPair, both CTAs' epilogues
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    if constexpr (kPair) {
      tmem_alloc_pair(tmem_slot, a.tmem_cols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(tmem_slot, a.tmem_cols);
      tmem_relinquish();
    }
    tc_fence_before_sync();
  }
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = ld_shared_b32(tmem_slot);
  // The peer's barriers are initialised before any of its loads, commits or
  // arrivals reach them.
  if constexpr (kPair) cluster_sync();

  // Nothing global has been touched yet: the kernel ahead in the stream may still
  // be running (programmatic launch), so wait for it here.
  grid_dependency_wait();

  if (warp < kLoaderWarps) {
    // ------------------------------------------------------------ Fetch --
    if (a.tma_load) {
      if (warp == 0 && lane == 0) {
        if constexpr (kGrouped) {
          for (int i = 0; i < g.n; ++i) tma_prefetch_map(&g.x[i]);
        } else {
          tma_prefetch_map(&tmap_x);
        }
        tma_prefetch_map(&tmap_w);
        int stage = 0;
        uint32_t phase = 0;
        uint32_t issued = 0, issued_parity = 0;
        // Bytes one CTA loads per stage; with kPair both CTAs' loads complete on
        // the first CTA's full barrier, which expects both.
        const int b_rows = kPair ? a.BN / 2 : a.BN;
        const uint32_t tx = static_cast<uint32_t>(kBM + b_rows) * 128u;
        for (long long tile = t_first; tile < a.num_tiles && !*abort_flag; tile += t_step) {
          int p, mb, nb;
          locate(tile, p, mb, nb);
          if (!CSA_CHECK(tile_ok(p, mb, nb), wd, kCheckTile)) break;
          const CUtensorMap* mx = map_x(p);
          bool ok = true;
          for (int kb = 0; kb < a.kblocks; ++kb) {
            if (!mbar_wait(empty_bar(stage), phase ^ 1u, wd, kSiteProducerEmpty)) {
              ok = false;
              break;
            }
            if (!kPair || rank == 0) mbar_arrive_expect_tx(full_bar(stage), kPair ? 2u * tx : tx);
            if (a.inject && tile == t_first && kb == 0) {
              issued &= ~(1u << stage);  // withheld: the MMA warp's wait must run out
            } else {
              if constexpr (kPair) {
                // This CTA's 128 rows of X and its half of the W tile's rows, both
                // completing on the first CTA's barrier.
                const uint32_t bar0 = mapa_shared(full_bar(stage), 0);
                tma_load_2d_pair(a_tile(stage), mx, bar0, kb * kBK, mb * kBM);
                tma_load_2d_pair(b_tile(stage), &tmap_w, bar0, kb * kBK,
                                 nb * a.BN + static_cast<int>(rank) * b_rows);
              } else {
                tma_load_2d(a_tile(stage), mx, full_bar(stage), kb * kBK, mb * kBM);
                tma_load_2d(b_tile(stage), &tmap_w, full_bar(stage), kb * kBK, nb * a.BN);
              }
              // (kPair: only the first CTA can see its loads land; the second CTA's
              // in-flight loads are covered by the teardown's grace period)
              if (!kPair || rank == 0) {
                issued |= 1u << stage;
                issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
              }
            }
            if (++stage == a.stages) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (!ok) break;
        }
        if (*abort_flag) {
          for (int s = 0; s < a.stages; ++s) {
            if (!(issued & (1u << s))) continue;
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_test(full_bar(s), (issued_parity >> s) & 1u) &&
                   globaltimer_ns() - t0 < a.wait_limit_ns) {
            }
          }
        }
      }
    } else if (kGrouped) {
      // (a group is always fetched by TMA)
    } else if (a.vec2) {
      // Asynchronous copies, kept up to `depth` stages ahead: a stage is handed to
      // the MMA warp (proxy fence + arrive) once this warp's copies into it have
      // completed, while later stages are still in flight.
      const int depth = a.load_depth;
      int stage = 0, oldest = 0, pending = 0, arrivals = 0;
      uint32_t phase = 0;
      bool aborted = false;
      for (long long tile = t_first; tile < a.num_tiles && !aborted; tile += t_step) {
        int p, mb, nb;
        locate(tile, p, mb, nb);
        for (int kb = 0; kb < a.kblocks; ++kb) {
          if (!mbar_wait_warp(empty_bar(stage), phase ^ 1u, wd, kSiteLoaderEmpty)) {
            aborted = true;
            break;
          }
          const int k = kb * kBK + 2 * static_cast<int>(lane);
          issue_block_async(a.X, a.M, mb * kBM, kBM, a.I, k, a_tile(stage), warp, lane);
          issue_block_async(a.W, a.H, nb * a.BN, a.BN, a.I, k, b_tile(stage), warp, lane);
          cp_async_commit();
          if (++pending == depth) {
            if (depth == 4) cp_async_wait<3>();
            else if (depth == 3) cp_async_wait<2>();
            else cp_async_wait<1>();
            fence_proxy_async_smem();  // completed generic-proxy writes -> tcgen05.mma
            __syncwarp();
            // (watchdog tests: the first stage is never handed over)
            if (lane == 0 && !(a.inject && arrivals == 0)) mbar_arrive(full_bar(oldest));
            ++arrivals;
            if (++oldest == a.stages) oldest = 0;
            --pending;
          }
          if (++stage == a.stages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      cp_async_wait<0>();
      fence_proxy_async_smem();
      __syncwarp();
      if (!aborted) {
        for (; pending > 0; --pending) {
          if (lane == 0 && !(a.inject && arrivals == 0)) mbar_arrive(full_bar(oldest));
          ++arrivals;
          if (++oldest == a.stages) oldest = 0;
        }
      }
    } else {
      int stage = 0;
      uint32_t phase = 0;
      for (long long tile = t_first; tile < a.num_tiles; tile += t_step) {
        int p, mb, nb;
        locate(tile, p, mb, nb);
        bool ok = true;
        for (int kb = 0; kb < a.kblocks; ++kb) {
          if (!mbar_wait_warp(empty_bar(stage), phase ^ 1u, wd, kSiteLoaderEmpty)) {
            ok = false;
            break;
          }
          const int k = kb * kBK + 2 * static_cast<int>(lane);
          load_block<false>(a.X, a.M, mb * kBM, kBM, a.I, k, a_tile(stage), warp, lane);
          load_block<false>(a.W, a.H, nb * a.BN, a.BN, a.I, k, b_tile(stage), warp, lane);
          fence_proxy_async_smem();  // generic smem writes -> visible to tcgen05.mma
          __syncwarp();
          // (watchdog tests: the first stage is never handed over)
          if (lane == 0 && !(a.inject && tile == blockIdx.x && kb == 0)) mbar_arrive(full_bar(stage));
          if (++stage == a.stages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
      }
    }
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------- Compute --
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      // With kPair only the pair's first CTA issues MMAs; the second waits for
      // their completion (the first CTA's drain commit reaches both).
      const bool issuer = !kPair || rank == 0;
      for (long long tile = t_first; issuer && tile < a.num_tiles; tile += t_step) {
        if (!mbar_wait(tempty_bar(acc), acc_phase ^ 1u, wd, kSiteMmaTmemEmpty)) break;
        tc_fence_after_sync();
        if (!CSA_CHECK(acc >= 0 && (acc + 1) * a.BN <= static_cast<int>(a.tmem_cols), wd,
                       kCheckTmem))
          break;
        const uint32_t d = tmem_base + static_cast<uint32_t>(acc * a.BN);
        bool ok = true;
        for (int kb = 0; kb < a.kblocks; ++kb) {
          if (!mbar_wait(full_bar(stage), phase, wd, kSiteMmaFull)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k) {
            const uint32_t off = static_cast<uint32_t>(k) * 32u;
            if constexpr (kPair)
              umma_bf16_pair(d, umma_desc_k_sw128(a_tile(stage) + off),
                             umma_desc_k_sw128(b_tile(stage) + off), a.idesc,
                             (kb > 0 || k > 0) ? 1u : 0u);
            else
              umma_bf16(d, umma_desc_k_sw128(a_tile(stage) + off),
                        umma_desc_k_sw128(b_tile(stage) + off), a.idesc,
                        (kb > 0 || k > 0) ? 1u : 0u);
          }
          if constexpr (kPair) umma_commit_pair_multicast(empty_bar(stage), 0x3);  // both CTAs
          else umma_commit(empty_bar(stage));
          if (++stage == a.stages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        if constexpr (kPair) umma_commit_pair_multicast(tfull_bar(acc), 0x3);
        else umma_commit(tfull_bar(acc));
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      if (issuer) {
        if constexpr (kPair) umma_commit_pair_multicast(drain_bar, 0x3);
        else umma_commit(drain_bar);
      }
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_test(drain_bar, 0) && globaltimer_ns() - t0 < a.wait_limit_ns) {
      }
    }
  } else {
    // -------------------------------------------------------- Writeback --
    const int q = static_cast<int>(warp & 3u);
    const uint32_t staging =
        base + a.off_staging + (warp - kFirstEpiWarp) * kStoreBufs * kBoxBytes;
    int acc = 0;
    uint32_t acc_phase = 0;
    uint32_t buf = 0;
    const int chunks = a.BN / 32;
    for (long long tile = t_first; tile < a.num_tiles; tile += t_step) {
      int p, mb, nb;
      locate(tile, p, mb, nb);
      if (!CSA_CHECK(tile_ok(p, mb, nb) &&
                         (acc + 1) * a.BN <= static_cast<int>(a.tmem_cols),
                     wd, kCheckTile))
        break;
      const int M = rows_of(p);
      if (!mbar_wait_warp(tfull_bar(acc), acc_phase, wd, kSiteEpilogueFull)) break;
      tc_fence_after_sync();
      const uint32_t tcol = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                            static_cast<uint32_t>(acc * a.BN);
      const int row0 = mb * kBM + q * 32;
      for (int c = 0; c < chunks; ++c) {
        uint32_t v[32];
        tmem_ld_32cols(tcol + static_cast<uint32_t>(c * 32), v);
        if (c == chunks - 1) {
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) {
            // (kPair: the accumulator is released on the pair's first CTA)
            if constexpr (kPair) mbar_arrive_cluster(mapa_shared(tempty_bar(acc), 0));
            else mbar_arrive(tempty_bar(acc));
          }
        }
        const int col0 = nb * a.BN + c * 32;
        if (row0 >= M || col0 >= a.H) continue;
        if (lane == 0) bulk_wait_read<kStoreBufs - 1>();
        __syncwarp();
        const uint32_t box = staging + buf * kBoxBytes;
        buf = (buf + 1u) & (kStoreBufs - 1u);
        stage_row_sw128(box, lane, v);
        if (a.tma_store) {
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(map_y(p), box, col0, row0);
            bulk_commit();
          }
        } else {
          __syncwarp();
          const int col = col0 + static_cast<int>(lane);
          float* ycol = y_of(p) + static_cast<size_t>(row0) * a.H + col;
          for (int rr = 0; rr < 32; ++rr) {
            const uint32_t val = staged_elem_sw128(box, static_cast<uint32_t>(rr), lane);
            if (row0 + rr < M && col < a.H)
              ycol[static_cast<size_t>(rr) * a.H] = __uint_as_float(val);
          }
        }
      }
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    // Only the stores' reads of shared memory must finish before the CTA exits;
    // their global writes complete before the grid does.
    if (lane == 0) bulk_wait_read<0>();
    __syncwarp();
  }

  __syncthreads();
  if constexpr (kPair) {
    // After a watchdog abort the second CTA cannot see its own loads land (they
    // complete on the first CTA's barrier): give any still in flight time to.
    if (*abort_flag && threadIdx.x == 0) {
      const uint64_t t0 = globaltimer_ns();
      while (globaltimer_ns() - t0 < 100000ull) {
      }
    }
    __syncthreads();
    // The peer's loads, commits and arrivals on this CTA are done.
    cluster_sync();
  }
  if (warp == kMmaWarp) {
    tc_fence_after_sync();
    if constexpr (kPair) tmem_dealloc_pair(tmem_base, a.tmem_cols);
    else tmem_dealloc(tmem_base, a.tmem_cols);
  }
}

// Rows of X [M, I], then of W [H, I], copied into rows of pitch P (I rounded
// up to a multiple of 64 elements) so that each copied row starts on a 128-byte
// boundary. Columns I..P-1 of a copied row are written as zeros (tensor maps
// with extent I never read them). One warp per row, one 16-byte destination
// chunk per lane and step, four steps' loads issued before their stores.
// `pairs`: the source rows are 4-byte aligned (I even, X and W 4-byte
// aligned) and are read as bf16 pairs, else one element at a time.
constexpr int kRealignThreads = 256;

// One row of I bf16 values copied by one warp into a row of pitch P (zeros in
// columns I..P-1), one 16-byte destination chunk per lane and step, four
// steps' loads issued before their stores.
__device__ __forceinline__ void realign_row(const uint16_t* __restrict__ src,
                                            uint16_t* __restrict__ dst, int I, int P, int pairs,
                                            int lane) {
  const int chunks = P / 8;
  for (int c0 = lane; c0 < chunks; c0 += 4 * 32) {
    uint32_t w[4][4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int k = (c0 + 32 * u) * 8;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int e = k + 2 * j;
        if (pairs) {
          w[u][j] = e < I ? __ldg(reinterpret_cast<const unsigned int*>(src + e)) : 0u;
        } else {
          const uint32_t lo = e < I ? __ldg(reinterpret_cast<const unsigned short*>(src + e)) : 0u;
          const uint32_t hi =
              e + 1 < I ? __ldg(reinterpret_cast<const unsigned short*>(src + e + 1)) : 0u;
          w[u][j] = lo | (hi << 16);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int c = c0 + 32 * u;
      if (c < chunks)
        *reinterpret_cast<uint4*>(dst + c * 8) = make_uint4(w[u][0], w[u][1], w[u][2], w[u][3]);
    }
  }
}

__global__ void __launch_bounds__(kRealignThreads)
    realign_rows_kernel(const uint16_t* __restrict__ X, const uint16_t* __restrict__ W,
                        uint16_t* __restrict__ Xp, uint16_t* __restrict__ Wp, int M, int H, int I,
                        int P, int pairs) {
  // X and W may be written by the kernel ahead in the stream (programmatic launch).
  grid_dependency_wait();
  const long long rows = static_cast<long long>(M) + H;
  const int lane = static_cast<int>(threadIdx.x & 31u);
  const long long warps_per_grid = static_cast<long long>(gridDim.x) * (kRealignThreads / 32);
  for (long long r = static_cast<long long>(blockIdx.x) * (kRealignThreads / 32) +
                     (threadIdx.x >> 5);
       r < rows; r += warps_per_grid) {
    const bool is_x = r < M;
    const uint16_t* src = is_x ? X + r * I : W + (r - M) * I;
    uint16_t* dst = is_x ? Xp + r * P : Wp + (r - M) * P;
    realign_row(src, dst, I, P, pairs, lane);
  }
}

// The same copy for the operands of a grouped call: up to kMaxGroup + 1 row
// ranges (W's rows and each X[g]'s), copied by one launch.
struct RealignSegments {
  const uint16_t* src[kMaxGroup + 1];
  uint16_t* dst[kMaxGroup + 1];
  long long first[kMaxGroup + 2];  // first row of range s in the launch's row list; [n] = all
  int n, I, P, pairs;
};

__global__ void __launch_bounds__(kRealignThreads)
    realign_segments_kernel(const __grid_constant__ RealignSegments g) {
  grid_dependency_wait();
  const int lane = static_cast<int>(threadIdx.x & 31u);
  const long long warps_per_grid = static_cast<long long>(gridDim.x) * (kRealignThreads / 32);
  for (long long r = static_cast<long long>(blockIdx.x) * (kRealignThreads / 32) +
                     (threadIdx.x >> 5);
       r < g.first[g.n]; r += warps_per_grid) {
    int lo = 0, hi = g.n - 1;  // the last range whose first row is <= r
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (g.first[mid] <= r) lo = mid;
      else hi = mid - 1;
    }
    const long long row = r - g.first[lo];
    realign_row(g.src[lo] + row * g.I, g.dst[lo] + row * g.P, g.I, g.P, g.pairs, lane);
  }
}

// Cost of a tiling: waves of `rows` x ceil(H / bn) work units over `slots`
// concurrent units (SMs, or clusters for CTA pairs), times the cost of one
// unit (~ bn plus a fixed per-tile overhead; each SM's share of a unit is a
// 128 x bn output tile in both forms).
long long tiling_cost(long long rows, int H, int bn, int slots) {
  const long long tiles = rows * ((H + bn - 1) / bn);
  return (tiles + slots - 1) / slots * (bn + 32);
}

// Tile width along H: the largest BN of least tiling cost, for `rows` rows of
// work units (128-row m-tiles, or pairs of them) over `slots` units at a time.
int choose_bn_tiles(long long rows, int H, int slots) {
  int best = 64;
  long long best_cost = -1;
  for (int bn : {256, 192, 128, 64}) {
    const long long cost = tiling_cost(rows, H, bn, slots);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = bn;
    }
  }
  return best;
}

// Clusters of two CTAs of `kernel` resident at once with `smem` bytes of
// dynamic shared memory each (its maximum already raised to that); 0 when none
// fit or the query fails.
int pair_clusters(const void* kernel, size_t smem, const DeviceInfo& dev) {
  struct Entry {
    const void* fn;
    int device;
    size_t smem;
    int clusters;
  };
  static std::mutex mu;
  static Entry cache[32];
  static int count = 0;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < count; ++i)
    if (cache[i].fn == kernel && cache[i].device == dev.device && cache[i].smem == smem)
      return cache[i].clusters;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 2;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();
    n = 0;
  }
  if (count < 32) cache[count++] = Entry{kernel, dev.device, smem, n};
  return n;
}

// TMEM columns for two BN-wide accumulators: an allocation is a power of two >= 32.
uint32_t tmem_cols_for(int BN) {
  uint32_t c = 32u;
  while (c < static_cast<uint32_t>(2 * BN)) c *= 2u;
  return c;
}

// Shared-memory plan: ring stages of 128 rows of X and b_rows rows of W (BN, or
// BN / 2 for a CTA pair), then staging, barriers and misc.
int plan_smem(DenseArgs& a, const DeviceInfo& dev, std::string& err, size_t& smem,
              int b_rows) {
  a.stage_bytes = static_cast<uint32_t>(kBM + b_rows) * 128u;
  const int fixed = kStagingBytes + 1024 + 1024;
  a.stages = std::min(CSA_DENSE_MAX_STAGES,
                      (dev.max_smem_optin - fixed) / static_cast<int>(a.stage_bytes));
  a.load_depth = std::min(a.stages, 4);
  if (a.stages < 2) {
    err = "dense_xwt: not enough shared memory";
    return CSA_ERR_UNSUPPORTED;
  }
  a.off_staging = static_cast<uint32_t>(a.stages) * a.stage_bytes;
  a.off_bars = a.off_staging + kStagingBytes;
  a.off_misc = a.off_bars + 8u * static_cast<uint32_t>(2 * a.stages + 5);
  smem = a.off_misc + 16 + 1024;
  return CSA_OK;
}

// Pitch (elements) of a realigned row: I rounded up to 64, so that every copied
// row starts on a 128-byte boundary and each 64-element TMA box row is one
// 128-byte line (with pitch I rounded up to 8 only, the rows are 16-byte
// aligned and every box row straddles two lines: the 32-problem sweep at
// I = 770 measured 188.0 us that way against 159.4 us with this pitch).
long long realigned_pitch(int I) { return (static_cast<long long>(I) + 63) / 64 * 64; }

// Rows that tensor maps can describe as they are: I * 2 a multiple of 16 and
// both operands 16-byte aligned.
bool rows_describable(const void* X, const void* W, int I) {
  return (static_cast<long long>(I) * 2) % 16 == 0 && reinterpret_cast<uintptr_t>(X) % 16 == 0 &&
         reinterpret_cast<uintptr_t>(W) % 16 == 0;
}

size_t round256(size_t n) { return (n + 255) / 256 * 256; }

}  // namespace

size_t dense_workspace_bytes(const void* X, const void* W, int M, int I, int H) {
  if (rows_describable(X, W, I)) return 0;
  const size_t P = static_cast<size_t>(realigned_pitch(I));
  return 256 + round256(static_cast<size_t>(M) * P * 2) + static_cast<size_t>(H) * P * 2;
}

void dense_tiling(int M, int H, int sms, bool tma_rows, int& bn, bool& pair) {
  const long long m_tiles = (static_cast<long long>(M) + kBM - 1) / kBM;
  const long long m_pairs = (m_tiles + 1) / 2;
  const int cluster_slots = sms / 2;
  bn = choose_bn_tiles(m_tiles, H, sms);
  pair = false;
  if (!tma_rows || cluster_slots < 1 || CSA_DENSE_SINGLE_PAIR == 0) return;
  const int bn_pair = choose_bn_tiles(m_pairs, H, cluster_slots);
  const long long cost_single = tiling_cost(m_tiles, H, bn, sms);
  const long long cost_pair = tiling_cost(m_pairs, H, bn_pair, cluster_slots);
  const long long pair_tiles = m_pairs * ((H + bn_pair - 1) / bn_pair);
  pair = CSA_DENSE_SINGLE_PAIR == 1 || cost_pair < cost_single ||
         (cost_pair == cost_single && pair_tiles >= 3LL * cluster_slots);
  if (pair) bn = bn_pair;
}

int dense_launch(float* Y, const void* X, const void* W, int M, int I, int H, void* workspace,
                 size_t ws_bytes, cudaStream_t stream, const DeviceInfo& dev, std::string& err) {
  const uintptr_t px = reinterpret_cast<uintptr_t>(X), pw = reinterpret_cast<uintptr_t>(W),
                  py = reinterpret_cast<uintptr_t>(Y);
  if (px % 2 || pw % 2 || py % 4) {
    err = "dense_xwt: X and W must be 2-byte aligned and Y 4-byte aligned";
    return CSA_ERR_ALIGN;
  }
  DenseArgs a{};
  a.M = M;
  a.I = I;
  a.H = H;
  a.m_tiles = (M + kBM - 1) / kBM;
  a.BN = choose_bn_tiles(a.m_tiles, H, dev.sm_count);
  a.kblocks = (I + kBK - 1) / kBK;
  a.tma_load = rows_describable(X, W, I) ? 1u : 0u;
  a.tma_store = ((static_cast<long long>(H) * 4) % 16 == 0 && py % 16 == 0) ? 1u : 0u;
  a.vec2 = (I % 2 == 0 && px % 4 == 0 && pw % 4 == 0) ? 1u : 0u;

  // Rows no tensor map can describe: copied first into the caller's workspace as
  // 16-byte-aligned rows (unless there is none, or the caller asked for the
  // loader-warp fetch), then fetched by TMA.
  const void* X_tma = X;
  const void* W_tma = W;
  long long pitch = I;
  bool realign = false;
  if (!a.tma_load && workspace && dense_fetch_mode() == CSA_DENSE_FETCH_AUTO) {
    const size_t need = dense_workspace_bytes(X, W, M, I, H);
    if (ws_bytes < need) {
      err = "dense_xwt_ws: " + std::to_string(need) + " bytes of workspace needed, " +
            std::to_string(ws_bytes) + " given";
      return CSA_ERR_WORKSPACE;
    }
    const long long P = realigned_pitch(I);
    uint8_t* p = static_cast<uint8_t*>(workspace);
    p += (256 - reinterpret_cast<uintptr_t>(p) % 256) % 256;
    X_tma = p;
    W_tma = p + round256(static_cast<size_t>(M) * P * 2);
    pitch = P;
    a.tma_load = 1u;
    realign = true;
  }
  // CTA pairs (256-row tiles, each SM loading half of the W tile) when the rows
  // are fetched by TMA and the pair tiling, counted in clusters of two, costs
  // less than single CTAs', or as much with three tiles or more per cluster.
  // (Measured with L2 flushed, I = 768, H = 3072: pairs 4-8 % faster from
  // M = 6144 up, within 1 us of single CTAs at 2-2.5 tiles per cluster, 2 us
  // slower where either form takes one wave.)
  auto* kernel_pair = dense_sm103a_kernel<false, true>;
  const long long m_pairs = (a.m_tiles + 1) / 2;
  bool pair = false;
  {
    int bn = 0;
    dense_tiling(M, H, dev.sm_count, a.tma_load != 0, bn, pair);
    if (pair) a.BN = bn;
  }
  a.X = static_cast<const uint16_t*>(X);
  a.W = static_cast<const uint16_t*>(W);
  a.Y = Y;
  a.status = dev.status_word;
  a.wait_limit_ns = wait_limit_ns();
  a.inject = take_inject() ? 1 : 0;

  size_t smem = 0;
  int clusters = 0;
  if (pair) {
    int rc = plan_smem(a, dev, err, smem, a.BN / 2);
    if (rc != CSA_OK) return rc;
    rc = set_max_dynamic_smem(reinterpret_cast<const void*>(kernel_pair), static_cast<int>(smem),
                              dev.device, err);
    if (rc != CSA_OK) {
      err = "dense_xwt: " + err;
      return rc;
    }
    // (at most one cluster per two of the SMs this call may use)
    clusters = std::min(pair_clusters(reinterpret_cast<const void*>(kernel_pair), smem, dev),
                        dev.sm_count / 2);
    if (clusters < 1) {
      pair = false;
      a.BN = choose_bn_tiles(a.m_tiles, H, dev.sm_count);
    }
  }
  a.n_tiles = (H + a.BN - 1) / a.BN;
  a.num_tiles = (pair ? m_pairs : static_cast<long long>(a.m_tiles)) * a.n_tiles;
  a.idesc = pair ? idesc_bf16_f32(2 * kBM, a.BN) : idesc_bf16_f32(kBM, a.BN);
  a.tmem_cols = tmem_cols_for(a.BN);
  if (!pair) {
    const int rc = plan_smem(a, dev, err, smem, a.BN);
    if (rc != CSA_OK) return rc;
  }

  CUtensorMap map_x, map_w, map_y;
  std::memset(&map_x, 0, sizeof map_x);
  std::memset(&map_w, 0, sizeof map_w);
  std::memset(&map_y, 0, sizeof map_y);
  if (a.tma_load) {
    const uint64_t dx[2] = {static_cast<uint64_t>(I), static_cast<uint64_t>(M)};
    const uint64_t dw[2] = {static_cast<uint64_t>(I), static_cast<uint64_t>(H)};
    const uint64_t st[1] = {static_cast<uint64_t>(pitch) * 2};
    const uint32_t bx[2] = {kBK, kBM};
    // (pairs: each CTA loads half of the W tile's rows)
    const uint32_t bw[2] = {kBK, static_cast<uint32_t>(pair ? a.BN / 2 : a.BN)};
    int rc = encode_tiled(&map_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, X_tma, dx, st, bx,
                          CU_TENSOR_MAP_SWIZZLE_128B, err);
    if (rc != CSA_OK) return rc;
    rc = encode_tiled(&map_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, W_tma, dw, st, bw,
                      CU_TENSOR_MAP_SWIZZLE_128B, err);
    if (rc != CSA_OK) return rc;
  }
  if (a.tma_store) {
    const uint64_t dy[2] = {static_cast<uint64_t>(H), static_cast<uint64_t>(M)};
    const uint64_t st[1] = {static_cast<uint64_t>(H) * 4};
    const uint32_t by[2] = {32, 32};
    int rc = encode_tiled(&map_y, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, Y, dy, st, by,
                          CU_TENSOR_MAP_SWIZZLE_128B, err);
    if (rc != CSA_OK) return rc;
  }

  if (!pair) {
    int rc = set_max_dynamic_smem(reinterpret_cast<const void*>(dense_sm103a_kernel<false>),
                                  static_cast<int>(smem), dev.device, err);
    if (rc != CSA_OK) {
      err = "dense_xwt: " + err;
      return rc;
    }
  }
  cudaError_t e;
  if (realign) {
    // The realigned copy, launched last of all so that a call that fails a
    // check launches nothing.
    const long long rows = static_cast<long long>(M) + H;
    const long long blocks = std::min<long long>(
        (rows + kRealignThreads / 32 - 1) / (kRealignThreads / 32), 16LL * dev.sm_count);
    e = launch_programmatic(realign_rows_kernel, static_cast<unsigned>(blocks), kRealignThreads,
                            0, stream, a.X, a.W, static_cast<uint16_t*>(const_cast<void*>(X_tma)),
                            static_cast<uint16_t*>(const_cast<void*>(W_tma)), M, H, I,
                            static_cast<int>(pitch), a.vec2 ? 1 : 0);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) {
      err = std::string("dense_xwt: launch: ") + cudaGetErrorString(e);
      return CSA_ERR_LAUNCH;
    }
  }
  if (pair) {
    const long long grid = 2 * std::min<long long>(a.num_tiles, clusters);
    e = launch_programmatic_cluster(kernel_pair, static_cast<unsigned>(grid), kThreads, smem,
                                    stream, 2u, map_x, map_w, map_y, a, DenseGroup<false>{});
  } else {
    const long long grid = std::min<long long>(a.num_tiles, dev.sm_count);
    e = launch_programmatic(dense_sm103a_kernel<false>, static_cast<unsigned>(grid), kThreads,
                            smem, stream, map_x, map_w, map_y, a, DenseGroup<false>{});
  }
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) {
    err = std::string("dense_xwt: launch: ") + cudaGetErrorString(e);
    return CSA_ERR_LAUNCH;
  }
  return CSA_OK;
}

}  // namespace csa

namespace csa {

// Y[g] = X[g] W^T for g < n: launches of up to kMaxGroup problems each when the
// rows of every X[g] and of W can be described by tensor maps (I * 2 % 16 == 0,
// 16-byte aligned), else one dense_launch per problem.
namespace {

bool group_rows_describable(const void* const* X, const void* W, int n, int I) {
  bool ok = (static_cast<long long>(I) * 2) % 16 == 0 && reinterpret_cast<uintptr_t>(W) % 16 == 0;
  for (int i = 0; ok && i < n; ++i) ok = reinterpret_cast<uintptr_t>(X[i]) % 16 == 0;
  return ok;
}

}  // namespace

size_t dense_grouped_workspace_bytes(const void* const* X, const void* W, const int* M, int n,
                                     int I, int H) {
  if (group_rows_describable(X, W, n, I)) return 0;
  const size_t P = static_cast<size_t>(realigned_pitch(I));
  size_t b = 256 + round256(static_cast<size_t>(H) * P * 2);
  for (int i = 0; i < n; ++i) b += round256(static_cast<size_t>(M[i]) * P * 2);
  return b;
}

int dense_grouped_launch(float* const* Y, const void* const* X, const void* W, const int* M, int n,
                         int I, int H, void* workspace, size_t ws_bytes, cudaStream_t stream,
                         const DeviceInfo& dev, std::string& err) {
  const bool tma_rows = group_rows_describable(X, W, n, I);
  bool tma_store = (static_cast<long long>(H) * 4) % 16 == 0;
  for (int i = 0; i < n; ++i) tma_store = tma_store && reinterpret_cast<uintptr_t>(Y[i]) % 16 == 0;
  const bool realign = !tma_rows && workspace && dense_fetch_mode() == CSA_DENSE_FETCH_AUTO;
  if (!tma_rows && !realign) {
    // No workspace (or the loader-warp fetch asked for): one dense_xwt per problem.
    for (int i = 0; i < n; ++i) {
      const int rc = dense_launch(Y[i], X[i], W, M[i], I, H, nullptr, 0, stream, dev, err);
      if (rc != CSA_OK) return rc;
    }
    return CSA_OK;
  }
  // Rows no tensor map can describe: W's and every X[g]'s rows are copied into the
  // workspace (W first, then the problems in order) as 16-byte-aligned rows of
  // pitch P, by one copy launch per group of problems, then read from there.
  long long pitch = I;
  const void* w_src = W;
  uint8_t* x_next = nullptr;
  int pairs = 0;
  if (realign) {
    const size_t need = dense_grouped_workspace_bytes(X, W, M, n, I, H);
    if (ws_bytes < need) {
      err = "dense_xwt_grouped_ws: " + std::to_string(need) + " bytes of workspace needed, " +
            std::to_string(ws_bytes) + " given";
      return CSA_ERR_WORKSPACE;
    }
    pitch = realigned_pitch(I);
    uint8_t* p = static_cast<uint8_t*>(workspace);
    p += (256 - reinterpret_cast<uintptr_t>(p) % 256) % 256;
    w_src = p;
    x_next = p + round256(static_cast<size_t>(H) * pitch * 2);
    pairs = I % 2 == 0 && reinterpret_cast<uintptr_t>(W) % 4 == 0;
    for (int i = 0; i < n; ++i) pairs = pairs && reinterpret_cast<uintptr_t>(X[i]) % 4 == 0;
  }
  CUtensorMap map_w;  // W's box depends on BN, chosen per launch below
  static thread_local DenseGroup<true> grp;  // 13 KB: kept off the stack
  static thread_local RealignSegments seg;
  const void* x_src[kMaxGroup];
  for (int first = 0; first < n; first += kMaxGroup) {
    const int cnt = std::min(kMaxGroup, n - first);
    if (realign) {
      std::memset(&seg, 0, sizeof seg);
      seg.I = I;
      seg.P = static_cast<int>(pitch);
      seg.pairs = pairs;
      long long rows = 0;
      if (first == 0) {
        seg.src[seg.n] = static_cast<const uint16_t*>(W);
        seg.dst[seg.n] = static_cast<uint16_t*>(const_cast<void*>(w_src));
        seg.first[seg.n++] = rows;
        rows += H;
      }
      for (int i = 0; i < cnt; ++i) {
        x_src[i] = x_next;
        seg.src[seg.n] = static_cast<const uint16_t*>(X[first + i]);
        seg.dst[seg.n] = reinterpret_cast<uint16_t*>(x_next);
        seg.first[seg.n++] = rows;
        rows += M[first + i];
        x_next += round256(static_cast<size_t>(M[first + i]) * pitch * 2);
      }
      seg.first[seg.n] = rows;
    } else {
      for (int i = 0; i < cnt; ++i) x_src[i] = X[first + i];
    }
    std::memset(&grp, 0, sizeof grp);
    grp.n = cnt;
    long long total = 0;
    for (int i = 0; i < cnt; ++i) {
      grp.mt_start[i] = static_cast<int>(total);
      grp.M[i] = M[first + i];
      grp.Y[i] = Y[first + i];
      total += (M[first + i] + kBM - 1) / kBM;
    }
    if (total >= (1LL << 30)) {
      err = "dense_xwt_grouped: too many row tiles in one group";
      return CSA_ERR_SHAPE;
    }
    grp.mt_start[cnt] = static_cast<int>(total);

    DenseArgs a{};
    a.M = 0;  // per problem: grp.M
    a.I = I;
    a.H = H;
    // Pairs of CTAs (clusters of two) walk tile pairs: adjacent m-tiles, one n-tile;
    // their tile width is chosen for pairs of m-tiles over clusters.
    bool pair = CSA_DENSE_PAIR != 0;
    a.BN = pair ? choose_bn_tiles((total + 1) / 2, H, std::max(1, dev.sm_count / 2))
                : choose_bn_tiles(total, H, dev.sm_count);
    a.m_tiles = static_cast<int>(total);
    a.n_tiles = (H + a.BN - 1) / a.BN;
    a.kblocks = (I + kBK - 1) / kBK;
    a.num_tiles = pair ? (total + 1) / 2 * a.n_tiles : total * a.n_tiles;
    a.tma_load = 1u;
    a.tma_store = tma_store ? 1u : 0u;
    a.vec2 = 0u;
    a.idesc = pair ? idesc_bf16_f32(2 * kBM, a.BN) : idesc_bf16_f32(kBM, a.BN);
    a.X = nullptr;
    a.W = static_cast<const uint16_t*>(W);
    a.Y = nullptr;
    a.status = dev.status_word;
    a.wait_limit_ns = wait_limit_ns();
    a.inject = take_inject() ? 1 : 0;
    a.tmem_cols = tmem_cols_for(a.BN);
    size_t smem = 0;
    int rc = plan_smem(a, dev, err, smem, pair ? a.BN / 2 : a.BN);
    if (rc != CSA_OK) return rc;

    // Clusters that can be resident at once with this much shared memory; none
    // (or an error) means no pairing.
    auto* kernel_pair = dense_sm103a_kernel<true, true>;
    int clusters = 0;
    if (pair) {
      rc = set_max_dynamic_smem(reinterpret_cast<const void*>(kernel_pair), static_cast<int>(smem),
                                dev.device, err);
      if (rc != CSA_OK) return rc;
      clusters = std::min(pair_clusters(reinterpret_cast<const void*>(kernel_pair), smem, dev),
                          dev.sm_count / 2);
      if (clusters < 1) {
        pair = false;
        a.BN = choose_bn_tiles(total, H, dev.sm_count);
        a.n_tiles = (H + a.BN - 1) / a.BN;
        a.tmem_cols = tmem_cols_for(a.BN);
        a.num_tiles = total * a.n_tiles;
        a.idesc = idesc_bf16_f32(kBM, a.BN);
        rc = plan_smem(a, dev, err, smem, a.BN);
        if (rc != CSA_OK) return rc;
      }
    }

    const uint64_t st_in[1] = {static_cast<uint64_t>(pitch) * 2};
    const uint32_t bx[2] = {kBK, kBM};
    // With pairs, each CTA loads (and multicasts) half of the W tile's rows.
    const uint32_t bw[2] = {kBK, static_cast<uint32_t>(pair ? a.BN / 2 : a.BN)};
    const uint64_t dw[2] = {static_cast<uint64_t>(I), static_cast<uint64_t>(H)};
    rc = encode_tiled(&map_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, w_src, dw, st_in, bw,
                      CU_TENSOR_MAP_SWIZZLE_128B, err);
    if (rc != CSA_OK) return rc;
    for (int i = 0; i < cnt; ++i) {
      const uint64_t dx[2] = {static_cast<uint64_t>(I), static_cast<uint64_t>(grp.M[i])};
      rc = encode_tiled(&grp.x[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, x_src[i], dx, st_in,
                        bx, CU_TENSOR_MAP_SWIZZLE_128B, err);
      if (rc != CSA_OK) return rc;
      if (a.tma_store) {
        const uint64_t dy[2] = {static_cast<uint64_t>(H), static_cast<uint64_t>(grp.M[i])};
        const uint64_t sy[1] = {static_cast<uint64_t>(H) * 4};
        const uint32_t by[2] = {32, 32};
        rc = encode_tiled(&grp.y[i], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, grp.Y[i], dy, sy, by,
                          CU_TENSOR_MAP_SWIZZLE_128B, err);
        if (rc != CSA_OK) return rc;
      }
    }
    rc = set_max_dynamic_smem(reinterpret_cast<const void*>(dense_sm103a_kernel<true>),
                              static_cast<int>(smem), dev.device, err);
    if (rc != CSA_OK) {
      err = "dense_xwt_grouped: " + err;
      return rc;
    }
    CUtensorMap unused;
    std::memset(&unused, 0, sizeof unused);
    cudaError_t e;
    if (realign) {
      // The copy, launched last of all the checks so that a failing call launches nothing.
      const long long rows = seg.first[seg.n];
      const long long blocks = std::min<long long>(
          (rows + kRealignThreads / 32 - 1) / (kRealignThreads / 32), 16LL * dev.sm_count);
      e = launch_programmatic(realign_segments_kernel, static_cast<unsigned>(blocks),
                              kRealignThreads, 0, stream, seg);
      if (e == cudaSuccess) e = cudaGetLastError();
      if (e != cudaSuccess) {
        err = std::string("dense_xwt_grouped: launch: ") + cudaGetErrorString(e);
        return CSA_ERR_LAUNCH;
      }
    }
    if (pair) {
      const long long grid = 2 * std::min<long long>(a.num_tiles, clusters);
      e = launch_programmatic_cluster(kernel_pair, static_cast<unsigned>(grid), kThreads, smem,
                                      stream, 2u, unused, map_w, unused, a, grp);
    } else {
      const long long grid = std::min<long long>(a.num_tiles, dev.sm_count);
      e = launch_programmatic(dense_sm103a_kernel<true>, static_cast<unsigned>(grid), kThreads,
                              smem, stream, unused, map_w, unused, a, grp);
    }
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) {
      err = std::string("dense_xwt_grouped: launch: ") + cudaGetErrorString(e);
      return CSA_ERR_LAUNCH;
    }
  }
  return CSA_OK;
}

}  // namespace csa
