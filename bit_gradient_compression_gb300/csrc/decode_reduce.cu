// Receiver average of Eqn (8) ("LoCo: Low-Bit Communication Adaptor for
// Large-scale Model Training", §3.3): decode W ranks' packed buckets and
// average them in fp32, rank order, one division by W.
//
// Two kernels, chosen per (bits, W) from measurements over W = 1..16 (2^30
// elements and the 7B bucket):
//  * k_decode_reduce (8-bit codes): CTA tiles staged by the cp.async pipeline;
//    every thread writes its E means into a shared-memory output tile and one
//    thread ships the tile with a bulk (TMA) store, so the output leaves in
//    full, contiguous lines.
//  * k_decode_reduce_wl (4-bit codes, where decoding every code costs more
//    issue slots per byte): every warp streams its own warp tiles through its
//    own pipeline stages (warp_pipeline) and never meets the CTA's other warps
//    at a barrier; each warp ships its tile's means with its own bulk store.
//    Up to 8 ranks: CTAs of 8 warps with 3 stages; beyond that the stages are
//    larger, and CTAs of 4 warps with 2 stages keep 4-5 CTAs resident.  The
//    CTAs per SM, where the steps are read, the output tiles per warp and the
//    order in which a warp takes its tiles are fitted per W (the knobs below,
//    each with its measurements); on large buckets a second instantiation
//    takes the tiles in groups of consecutive ones, chosen at launch.
#include "receiver_common.cuh"

namespace loco {

#ifndef LOCO_REDUCE_ELEMS
#define LOCO_REDUCE_ELEMS(bits) (64 / (bits))  // elements per thread: 8 code bytes per rank
#endif
#ifndef LOCO_REDUCE_MIN_CTAS
#define LOCO_REDUCE_MIN_CTAS 3  // CTAs per SM the stage counts are fitted for
#endif
#ifndef LOCO_REDUCE_CTA_4BIT
#define LOCO_REDUCE_CTA_4BIT(w) 0  // rank counts whose 4-bit codes take the CTA-tile kernel (none)
#endif
#ifndef LOCO_REDUCE_STAGES8
// Stages of the 8-bit kernel: two below 7 ranks; from 7 ranks one stage per
// CTA (each CTA loads, then computes, and the CTAs of an SM overlap one
// another) measured faster (W = 12: 86 % -> 101 %, W = 7: 95 % -> 99 %;
// W = 2: 95 % -> 88 %, W = 6: 98 % -> 97 %).
#define LOCO_REDUCE_STAGES8(w) ((w) >= 7 ? 1 : 2)
#endif
#ifndef LOCO_REDUCE_STAGES4
#define LOCO_REDUCE_STAGES4 3
#endif
#ifndef LOCO_REDUCE_WL_MIN_CTAS
// CTAs per SM the warp-local kernel is fitted for up to LOCO_REDUCE_WL_BULK_MAX_W
// ranks: four at W = 3..6 (its registers capped at 64; 0.89-0.98 of the copy
// rate at 2^30 elements against 0.83-0.91 with three), three at W = 7, 8 (four
// leaves room for only two stages there: 0.82 / 0.94 against 0.91 / 0.97).
// W = 1, 2 need fewer than 64 registers and run four either way.
#define LOCO_REDUCE_WL_MIN_CTAS(w) ((w) >= 3 && (w) <= 6 ? 4 : LOCO_REDUCE_MIN_CTAS)
#endif
#ifndef LOCO_REDUCE_WL_OUT_BUFS
// Output tiles per warp with bulk stores: two (one store in flight while the
// next tile's means are written) measured faster at W = 2 (0.96 of the copy
// rate against 0.94), slower at W = 1 and W = 4..8.
#define LOCO_REDUCE_WL_OUT_BUFS(w) ((w) == 2 ? 2 : 1)
#endif
#ifndef LOCO_REDUCE_WL_GROUP
// Consecutive warp tiles each warp of the warp-local kernel takes in turn on
// buckets of at least LOCO_REDUCE_WL_GROUP_MIN_TILES(W) warp tiles per warp of
// the resident grid (smaller buckets, and W = 1, 2, 6: tiles gw, gw + nw,
// gw + 2 nw, ...; G: tiles G gw .. G gw + G-1, then the group nw further on).
// Over many tiles the warps drift apart, and the reads of one DRAM page of a
// rank's codes then arrive from warps far apart in time; a group keeps a
// page's reads within one warp.  Measured against the plain order (fraction of
// the copy rate; 2^28 / 2^30 elements / the 6.7G-element Llama-2-7B bucket):
// W = 16 0.90 -> 0.91 at 2^30, 0.85 -> 0.91 on the 7B bucket; W = 3 0.904 ->
// 0.916 / 0.928 -> 0.937 / 0.930 -> 0.948; W = 7 0.904 -> 0.917 / 0.930 ->
// 0.942 / 0.927 -> 0.948; W = 4, 5 the same or better.  W = 8: 0.952 -> 0.960
// on the 7B bucket (3608 tiles per warp; the same at 2^32, 2299) but 0.968 ->
// 0.953 at 2^30 (575), hence its higher threshold.  W = 2 (two output tiles
// per warp) 0.967 -> 0.881 and W = 6 0.935 -> 0.920 on the 7B bucket.
#define LOCO_REDUCE_WL_GROUP(w) ((w) == 1 || (w) == 2 || (w) == 6 ? 1 : 8)
#endif
#ifndef LOCO_REDUCE_WL_GROUP_MIN_TILES
#define LOCO_REDUCE_WL_GROUP_MIN_TILES(w) ((w) == 8 ? 2048 : 64)
#endif
#ifndef LOCO_REDUCE_WL_BULK_MAX_W
#define LOCO_REDUCE_WL_BULK_MAX_W 8  // largest rank count of the warp-local kernel with bulk output stores
#endif
#ifndef LOCO_REDUCE_WL_STAGES_BULK
#define LOCO_REDUCE_WL_STAGES_BULK(w) 3  // stages up to LOCO_REDUCE_WL_BULK_MAX_W ranks (5 or 6 at W <= 4: no faster)
#endif
#ifndef LOCO_REDUCE_WL_WARPS_HI
#define LOCO_REDUCE_WL_WARPS_HI 4  // warps per CTA of the warp-local kernel beyond LOCO_REDUCE_WL_BULK_MAX_W ranks
#endif
#ifndef LOCO_REDUCE_WL_BULK_HI
#define LOCO_REDUCE_WL_BULK_HI 1  // bulk output stores beyond LOCO_REDUCE_WL_BULK_MAX_W ranks
#endif
#ifndef LOCO_REDUCE_WL_MIN_CTAS_HI
#define LOCO_REDUCE_WL_MIN_CTAS_HI(w) ((w) <= 11 ? 5 : 4)
#endif
#ifndef LOCO_REDUCE_WL_STAGES_HI
#define LOCO_REDUCE_WL_STAGES_HI 2
#endif
#ifndef LOCO_REDUCE_WL_STEPS_SMEM
// Rank counts whose tiles stage their steps with the codes (cp.async) instead
// of reading them one tile ahead into registers: measured faster at W = 1, 3,
// 7 and W > 8 (W = 3: 0.88 -> 0.93 of the copy rate, W = 7: 0.91 -> 0.93),
// slower at W = 2, 4, 5, 8 (0.95 -> 0.90 at W = 2), the same at W = 6.
#define LOCO_REDUCE_WL_STEPS_SMEM(w) ((w) == 1 || (w) == 3 || (w) == 7 || (w) > 8)
#endif

template <int BITS, int W>
constexpr bool use_warp_local() {
  return BITS == 4 && !(LOCO_REDUCE_CTA_4BIT(W));
}

// ---------------------------------------------------------------------------
// CTA-tile kernel with a bulk output store per tile.
// ---------------------------------------------------------------------------
template <int BITS, int W, int E>
struct DecodeSmem {
  static constexpr size_t kOut = size_t(kThreads) * E * 4;  // one output tile
  static constexpr int S =
      fit_stages<BITS, W, E, 0>(BITS == 8 ? LOCO_REDUCE_STAGES8(W) : LOCO_REDUCE_STAGES4, kOut, LOCO_REDUCE_MIN_CTAS);
  static constexpr size_t kBytes = size_t(S) * Tile<BITS, W, E, 0>::kBytes + kOut;
};

template <int BITS, int W, int E, int S>
__global__ void __launch_bounds__(kThreads) k_decode_reduce(const ReduceArgs a, int log2_block) {
  extern __shared__ __align__(16) uint8_t sm[];
  using TL = Tile<BITS, W, E, 0>;
  float* out = reinterpret_cast<float*>(sm + size_t(S) * TL::kBytes);
  const float* none[1] = {nullptr};
  const bool leader = threadIdx.x == 0;
  tile_pipeline<BITS, W, E, 0, S>(
      none, a.ranks, a.n, log2_block,
      [&](const TL& tl, int64_t) {
        float mean[E];
        tile_mean<BITS, W, E, 0>(tl, threadIdx.x, log2_block, a.ranks.neg_zero, mean);
        float4* o = reinterpret_cast<float4*>(out + threadIdx.x * E);
#pragma unroll
        for (int q = 0; q < E / 4; ++q) o[q] = make_float4(mean[4 * q], mean[4 * q + 1], mean[4 * q + 2], mean[4 * q + 3]);
        fence_smem_to_async_proxy();  // make the tile visible to the bulk copy
      },
      [&](int64_t e0) {
        float mean[E];
        decode_mean<BITS, W, E>(a.ranks, e0, e0 >> log2_block, mean);
        store_vec<E>(a.mean, e0, a.n, e0 + E <= a.n, mean);
      },
      // before a tile is published: the previous tile's bulk store has read `out`
      [&](int64_t) {
        if (leader) bulk_wait_read_all();
      },
      // after every thread wrote `out`: one thread ships it
      [&](int64_t tile) {
        if (leader) {
          bulk_store(a.mean + tile * TL::T, out, uint32_t(TL::T * 4));
          bulk_commit();
        }
      });
  if (leader) bulk_wait_all();
}

// ---------------------------------------------------------------------------
// Warp-local kernel: every warp streams its own warp tiles of WT = 32*E
// elements through S stages of its own shared memory (warp_pipeline).  A stage
// holds the W ranks' packed codes of one warp tile (W * WT*BITS/8 bytes, rank
// major), copied as 16-byte pieces by the warp's lanes.  The W steps a lane
// needs (one block per lane: E <= block) are read one tile ahead into
// registers, or, for the rank counts LOCO_REDUCE_WL_STEPS_SMEM names, copied
// into the stage after the codes as 8-byte pieces.  With BULK each warp writes
// its tile's means into one of its own OUT_BUFS output tiles in shared memory
// (in turn) and lane 0 ships it with one bulk (TMA) store; a tile's means go
// into an output tile only after the store that last shipped it has read it.
// ---------------------------------------------------------------------------
template <int BITS, int W, int E, bool BULK, int WARPS, bool STEPS_SMEM, int OUT_BUFS = 1>
struct WarpTile {
  static constexpr int kOutBufs = OUT_BUFS;
  static_assert(OUT_BUFS == 1 || OUT_BUFS == 2, "one or two output tiles per warp");
  static constexpr int kWarps = WARPS;
  static constexpr bool kStepsSmem = STEPS_SMEM;
  static constexpr int WT = 32 * E;                      // elements per warp tile
  static constexpr int CB = WT * BITS / 8;               // code bytes per rank and warp tile
  static constexpr int kPieces = CB / 16;                // 16-byte pieces per rank
  static constexpr int kJobs = (W * kPieces + 31) / 32;  // pieces per lane
  static constexpr int kStepsMax = WT / 64;                  // steps per rank and tile, smallest block
  static constexpr size_t kStepBytes = STEPS_SMEM ? size_t(W) * kStepsMax * 4 : 0;
  static constexpr size_t kStage = size_t(W) * CB + kStepBytes;
  static constexpr size_t kOut = BULK ? size_t(OUT_BUFS) * WT * 4 : 0;  // per-warp output tiles
  static_assert(CB % 16 == 0, "whole 16-byte pieces");
  static constexpr size_t bytes(int st) { return size_t(kWarps) * (st * kStage + kOut); }
  // Largest stage count <= want (>= 2) for which min_ctas CTAs fit on one SM.
  static constexpr int stages(int want, int min_ctas) {
    int st = want;
    while (st > 2 && (size_t(min_ctas) * (bytes(st) + 1024) > size_t(228) * 1024 || bytes(st) > size_t(227) * 1024))
      --st;
    return st;
  }
};

// Configuration of the warp-local kernel for W ranks: CTA size, output path,
// stage count, and the CTAs per SM its shared memory and registers are fitted for.
template <int BITS, int W, int E>
struct WarpLocalConfig {
  static constexpr bool kLow = W <= LOCO_REDUCE_WL_BULK_MAX_W;
  static constexpr int kWarps = kLow ? 8 : LOCO_REDUCE_WL_WARPS_HI;
  static constexpr bool kBulk = kLow ? true : (LOCO_REDUCE_WL_BULK_HI != 0);
  static constexpr int kMinCtas = kLow ? LOCO_REDUCE_WL_MIN_CTAS(W) : LOCO_REDUCE_WL_MIN_CTAS_HI(W);
  using WTL = WarpTile<BITS, W, E, kBulk, kWarps, bool(LOCO_REDUCE_WL_STEPS_SMEM(W)),
                      kBulk ? LOCO_REDUCE_WL_OUT_BUFS(W) : 1>;
  static constexpr int S = WTL::stages(kLow ? LOCO_REDUCE_WL_STAGES_BULK(W) : LOCO_REDUCE_WL_STAGES_HI, kMinCtas);
  static constexpr size_t kSmem = WTL::bytes(S);
  static_assert(kSmem <= 227 * 1024, "staging area exceeds one CTA's shared memory");
};

template <int BITS, int W, int E, int G>
__global__ void __launch_bounds__(WarpLocalConfig<BITS, W, E>::kWarps * 32, WarpLocalConfig<BITS, W, E>::kMinCtas)
    k_decode_reduce_wl(const ReduceArgs a, int log2_block) {
  extern __shared__ __align__(16) uint8_t sm[];
  using CF = WarpLocalConfig<BITS, W, E>;
  using WTL = typename CF::WTL;
  constexpr int S = CF::S;
  constexpr bool BULK = CF::kBulk;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  uint8_t* wsm = sm + size_t(warp) * S * WTL::kStage;
  float* wout = reinterpret_cast<float*>(sm + size_t(WTL::kWarps) * S * WTL::kStage) + size_t(warp) * WTL::kOutBufs * WTL::WT;
  [[maybe_unused]] int ob = 0;  // with two output tiles: the one the next tile's means go to
  const int64_t gw = int64_t(blockIdx.x) * WTL::kWarps + warp;
  const int64_t nw = int64_t(gridDim.x) * WTL::kWarps;
  const int64_t ntiles = a.n / WTL::WT;

  // This lane's pieces of every tile: piece p = lane + 32*j is piece p % kPieces
  // of rank p / kPieces; it lands at byte 16*p of the stage (rank-major, CB =
  // 16*kPieces) and comes from the same offset of every tile (plus tile*CB).
  const uint8_t* src[WTL::kJobs];
#pragma unroll
  for (int j = 0; j < WTL::kJobs; ++j) {
    const int p = lane + 32 * j;
    src[j] = (p < W * WTL::kPieces) ? a.ranks.codes[p / WTL::kPieces] + 16 * (p % WTL::kPieces) : nullptr;
  }
  // With the steps staged: a tile's nsc steps per rank are 8-byte pieces
  // (nsc/2 per rank, W*nsc/2 <= 64 in all), at most two per lane.
  const int nsc = WTL::WT >> log2_block;
  const float* ssrc[2];
  uint32_t sdst[2];
  bool sval[2];
  if constexpr (WTL::kStepsSmem) {
    const int half = nsc >> 1;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int p = lane + 32 * j;
      sval[j] = p < W * half;
      const int w = sval[j] ? p / half : 0, k = sval[j] ? p % half : 0;
      ssrc[j] = a.ranks.scales[w] + 2 * k;
      sdst[j] = uint32_t(W * WTL::CB + (w * WTL::kStepsMax + 2 * k) * 4);
    }
  }
  auto issue = [&](uint8_t* st, int64_t tile) {
#pragma unroll
    for (int j = 0; j < WTL::kJobs; ++j)
      if ((W * WTL::kPieces) % 32 == 0 || lane + 32 * j < W * WTL::kPieces)
        cp_async16(st + 16 * (lane + 32 * j), src[j] + tile * WTL::CB);
    if constexpr (WTL::kStepsSmem) {
#pragma unroll
      for (int j = 0; j < 2; ++j)
        if (sval[j]) cp_async8(st + sdst[j], ssrc[j] + tile * nsc);
    }
  };
  // The tile this warp takes after `tile`.
  constexpr int kGroup = G;
  [[maybe_unused]] auto next_tile = [&](int64_t tile) {
    if constexpr (kGroup == 1) return tile + nw;
    else return (tile % kGroup != kGroup - 1) ? tile + 1 : tile + 1 + (nw - 1) * kGroup;
  };
  // Steps of this lane's block for every rank, one tile ahead in registers.
  float sc[W];
  auto load_steps = [&](float (&s)[W], int64_t tile) {
    const int64_t blk = (tile * WTL::WT + int64_t(lane) * E) >> log2_block;
#pragma unroll
    for (int w = 0; w < W; ++w) s[w] = __ldg(a.ranks.scales[w] + blk);
  };
  if constexpr (!WTL::kStepsSmem)
    if (gw * kGroup < ntiles) load_steps(sc, gw * kGroup);
  warp_pipeline<S, kGroup>(wsm, WTL::kStage, gw, nw, ntiles, issue, [&](const uint8_t* st, int64_t tile) {
    float nsc_[W];
    if constexpr (WTL::kStepsSmem) {
      const float* ss = reinterpret_cast<const float*>(st + W * WTL::CB) + ((lane * E) >> log2_block);
#pragma unroll
      for (int w = 0; w < W; ++w) sc[w] = ss[w * WTL::kStepsMax];
    } else {
      if (next_tile(tile) < ntiles) load_steps(nsc_, next_tile(tile));
    }
    ChunkCodes<BITS, E> cw[W];
#pragma unroll
    for (int w = 0; w < W; ++w) cw[w].load_shared(st + w * WTL::CB + lane * (E * BITS / 8));
    float mean[E];
    mean_of_codes<BITS, W, E>(cw, sc, a.ranks.neg_zero, mean);
    if constexpr (BULK) {
      float* ot = wout;  // this tile's output tile
      if constexpr (WTL::kOutBufs == 1) {
        if (lane == 0) bulk_wait_read_all();  // the previous tile's store has read the output tile
      } else {
        ot = wout + ob * WTL::WT;
        ob ^= 1;
        if (lane == 0) bulk_wait_read<1>();  // the store before the previous one has read this output tile
      }
      __syncwarp();
      float4* o = reinterpret_cast<float4*>(ot + lane * E);
#pragma unroll
      for (int q = 0; q < E / 4; ++q) o[q] = make_float4(mean[4 * q], mean[4 * q + 1], mean[4 * q + 2], mean[4 * q + 3]);
      fence_smem_to_async_proxy();  // this lane's means visible to the bulk copy
      __syncwarp();
      if (lane == 0) {
        bulk_store(a.mean + tile * WTL::WT, ot, uint32_t(WTL::WT * 4));
        bulk_commit();
      }
    } else {
      store_vec<E>(a.mean, tile * WTL::WT + int64_t(lane) * E, a.n, true, mean);
    }
    if constexpr (!WTL::kStepsSmem) {
#pragma unroll
      for (int w = 0; w < W; ++w) sc[w] = nsc_[w];
    }
  });
  if constexpr (BULK)
    if (lane == 0) bulk_wait_all();
  // Elements past the last full warp tile: one warp, straight from global memory.
  if (ntiles * WTL::WT < a.n && gw == ntiles % nw) {
    const int64_t e0 = ntiles * WTL::WT + int64_t(lane) * E;
    if (e0 < a.n) {
      float mean[E];
      decode_mean<BITS, W, E>(a.ranks, e0, e0 >> log2_block, mean);
      store_vec<E>(a.mean, e0, a.n, e0 + E <= a.n, mean);
    }
  }
}

// Grid of the warp-local kernel with tile groups of G: resident CTAs, at most
// one per CTA-worth of elements.
template <int BITS, int W, int E, int G>
cudaError_t wl_grid(const ReduceArgs& a, int* grid) {
  using CF = WarpLocalConfig<BITS, W, E>;
  static GridCache cache;
  int cap = 0;
  const cudaError_t e = grid_cap(cache, reinterpret_cast<const void*>(&k_decode_reduce_wl<BITS, W, E, G>),
                                 CF::kWarps * 32, CF::kSmem, &cap);
  if (e == cudaSuccess) *grid = clamp_grid(a.n, CF::kWarps * 32 * E, cap);
  return e;
}

template <int BITS, int W, int E, int G>
cudaError_t launch_wl(const ReduceArgs& a, int grid, cudaStream_t s) {
  using CF = WarpLocalConfig<BITS, W, E>;
  k_decode_reduce_wl<BITS, W, E, G><<<grid, CF::kWarps * 32, CF::kSmem, s>>>(a, ilog2_int(a.block));
  return cudaGetLastError();
}

template <int BITS>
struct DecodeLaunch {
  template <int W>
  struct F {
    static cudaError_t run(const ReduceArgs& a, cudaStream_t s) {
      constexpr int E = LOCO_REDUCE_ELEMS(BITS);
      if constexpr (use_warp_local<BITS, W>()) {
        using CF = WarpLocalConfig<BITS, W, E>;
        constexpr int G = LOCO_REDUCE_WL_GROUP(W);
        int grid = 0;
        cudaError_t e = wl_grid<BITS, W, E, 1>(a, &grid);
        if (e != cudaSuccess) return e;
        if constexpr (G > 1) {
          // warp tiles per warp of the resident grid
          const int64_t per_warp = (a.n / CF::WTL::WT) / (int64_t(grid) * CF::kWarps);
          if (per_warp >= LOCO_REDUCE_WL_GROUP_MIN_TILES(W)) {
            e = wl_grid<BITS, W, E, G>(a, &grid);
            if (e != cudaSuccess) return e;
            return launch_wl<BITS, W, E, G>(a, grid, s);
          }
        }
        return launch_wl<BITS, W, E, 1>(a, grid, s);
      } else {
        using SM = DecodeSmem<BITS, W, E>;
        static_assert(SM::kBytes <= 227 * 1024, "staging area exceeds one CTA's shared memory");
        static GridCache cache;
        int cap = 0;
        const cudaError_t e = grid_cap(cache, reinterpret_cast<const void*>(&k_decode_reduce<BITS, W, E, SM::S>),
                                       kThreads, SM::kBytes, &cap);
        if (e != cudaSuccess) return e;
        const int grid = clamp_grid(a.n, kThreads * E, cap);
        k_decode_reduce<BITS, W, E, SM::S><<<grid, kThreads, SM::kBytes, s>>>(a, ilog2_int(a.block));
        return cudaGetLastError();
      }
    }
  };
};

cudaError_t launch_decode_reduce(const ReduceArgs& a, cudaStream_t s) {
  return a.bits == 4 ? dispatch_w<DecodeLaunch<4>::F>(a.W, a, s) : dispatch_w<DecodeLaunch<8>::F>(a.W, a, s);
}

}  // namespace loco
