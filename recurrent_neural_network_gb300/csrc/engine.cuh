// engine.cuh -- the two GEMM mainloops every product of the recurrent path
// runs on, both computing   D[m][n] = sum_k A(m,k) * B(n,k)   tile by tile and
// handing each finished tile to an epilogue functor:
//
//  * tc_gemm_kernel: bf16 operands on the fifth-generation tensor cores.
//    One warp issues TMA tile loads into a STAGES-deep shared-memory ring
//    (128-byte swizzle), one thread issues tcgen05.mma into a double-buffered
//    TMEM accumulator, four warps run the epilogue straight out of TMEM while
//    the next tile's MMAs proceed.  Operands may be K-major or MN-major (the
//    transposed products of the backward pass need the latter).  Tiles are
//    128 x BN, K step 64; the grid is persistent over tiles and split-K ranges.
//  * simt_gemm_kernel: fp32 FFMA (no TF32) for the fp32 storage mode, with
//    compensated (error-free transformation) accumulation.
//
// Epilogue functors implement
//   template <class Acc> __device__ void operator()(const TileCoord&, int row, const Acc&) const
// where `row` is the row inside the tile owned by the calling thread and
// Acc::load16(col, v) returns 16 consecutive accumulator columns of that row.
// All threads of a warp call load16 together (TMEM loads are warp-collective).
#pragma once

#include <type_traits>

#include <cuda.h>

#include "common.cuh"
#include "tc.cuh"

namespace rnn {

struct GemmGeom {
  int M, N, K;
  int m_tiles, n_tiles, splits;
  int kb_total, kb_per_split;  // K blocks of 64 (tcgen05) or 16 (SIMT)
  int num_tiles;               // m_tiles * n_tiles * splits
  int a_mn, b_mn;              // operand majorness (1 = MN-major)
  int a3, b3;                  // MN-major operand with a 3-D map: all 64-wide blocks of a tile in one load
  uint64_t limit_ns;           // bound on every pipeline wait
  int* err;                    // device error word
  int cluster;                 // > 1: the split-K CTAs of a tile form one thread-block cluster
  int nfast;                   // tile order: n-tiles fastest
  int pdl;                     // launched as a programmatic dependent: wait before touching produced data
  int static_op;               // operand no earlier kernel writes (0 none, 1 A, 2 B): its first STAGES
                               // blocks of the first tile are loaded before that wait
  // Several dependent steps in one launch (CTA pairs, one tile per pair and step; steps > 1): tile
  // index = step * tiles_per_step + tile of the step, the B rows of step s start b_step_rows * s
  // further, and a pair loads the B operand of step s > 0 only once step_cnt[s - 1] has reached
  // step_want (the epilogue arrives on step_cnt[s] when its stores of step s are complete).
  int steps, tiles_per_step, b_step_rows;
  unsigned int* step_cnt;
  unsigned int step_want;
};

struct TileCoord {
  int m0, n0;       // first row / column of the tile
  int mt, nt;       // tile indices
  int step;         // step of a launch over several dependent steps (GemmGeom::steps), else 0
  int split, splits;
  int part, parts;  // this thread's share of the tile's columns (epilogues with 8 warps: 2 parts)
  int* scratch;     // 8 ints of shared memory for the epilogue warps (tcgen05 only)
  // cluster split-K (tcgen05, cluster > 1): the CTA's stage buffers reused as a
  // float tile for the reduction, and two cluster-wide barriers
  int cluster;     // number of CTAs that reduce together (the K splits)
  int peer_base;   // cluster rank of split 0 of this CTA's reduction group
  int peer_stride; // rank distance between consecutive splits of the group
  float* red;
  uint64_t* red_full;
  uint64_t* red_done;
  uint64_t* aux;  // [3]
};

// Epilogues that declare a Stash type can stage their global inputs while the
// MMAs run: stage() copies them into the CTA's idle second TMEM accumulator
// (and into registers held in the Stash) before the accumulator is complete,
// run_staged() then reads them from there.  The engine uses it when a CTA has
// exactly one tile, so that the second accumulator stays unused.
template <class E, class = void>
struct EpiStaged {
  static constexpr bool value = false;
  using Stash = int;
};
template <class E>
struct EpiStaged<E, std::void_t<typename E::Stash>> {
  static constexpr bool value = true;
  using Stash = typename E::Stash;
};

// Number of epilogue warps: 4 (one per TMEM lane quadrant) unless the
// epilogue declares kWarps = 8, in which case two warps share each quadrant
// and split the tile's columns (TileCoord::part of TileCoord::parts).  More
// warps hide the latency of the epilogue's dependent arithmetic and stores.
template <class E, class = void>
struct EpiWarps {
  static constexpr int value = 4;
};
template <class E>
struct EpiWarps<E, std::void_t<decltype(E::kWarps)>> {
  static constexpr int value = E::kWarps;
};
// FFMA engine: threads per tile row in the epilogue (1 unless the epilogue
// declares kSimtShares and shares out a row's elements by TileCoord::part)
template <class E, class = void>
struct EpiSimtShares {
  static constexpr int value = 1;
};
template <class E>
struct EpiSimtShares<E, std::void_t<decltype(E::kSimtShares)>> {
  static constexpr int value = E::kSimtShares;
};

// Epilogues with a tail_prefetch(const TileCoord&, int bn) member get it
// called by the TMA producer thread of the single-CTA engine once it has
// issued the last loads of the CTA's last tile: a few pipeline stages before
// the MMAs finish, late enough that what it pulls into L2 is not evicted by
// the operand stream (e.g. the inputs of the kernel that follows).
template <class E, class = void>
struct EpiTail {
  static constexpr bool value = false;
};
template <class E>
struct EpiTail<E, std::void_t<decltype(&E::tail_prefetch)>> {
  static constexpr bool value = true;
};

struct TmemAcc {
  uint32_t taddr;
  __device__ __forceinline__ void load16(int col, float* v) const { tc::tmem_load16(taddr + col, v); }
  // 32 columns of this accumulator and of `other` with a single wait
  __device__ __forceinline__ void load32_with(const TmemAcc& other, int col, float* v, float* w) const {
    tc::tmem_load32x2(taddr + col, other.taddr + col, v, w);
  }
};

struct SmemAcc {
  const float* row;
  __device__ __forceinline__ void load16(int col, float* v) const {
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = row[col + i];
  }
};

// Launches over several dependent steps: the step of a tile index, the tile
// index within its step left in `tile`.
__device__ __forceinline__ int step_of(const GemmGeom& g, int& tile) {
  if (g.steps <= 1) return 0;
  const int s = tile / g.tiles_per_step;
  tile -= s * g.tiles_per_step;
  return s;
}

// Bounded wait until *cnt >= want (acquire); gives up when the CTA aborts, and
// on timeout records DEV_TIMEOUT_STEP and marks the CTA aborted.
__device__ __forceinline__ bool wait_step(const unsigned int* cnt, unsigned int want, volatile int* abort_flag,
                                          int* err, uint64_t limit_ns) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(cnt) : "memory");
  if (v >= want) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(cnt) : "memory");
    if (v >= want) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > limit_ns) {
      raise_error(err, DEV_TIMEOUT_STEP);
      *abort_flag = 1;
      return false;
    }
  }
}

__device__ __forceinline__ void decode_tile(const GemmGeom& g, int tile, int& mt, int& nt, int& split) {
  split = tile % g.splits;
  const int mn = tile / g.splits;
  if (g.nfast) {
    nt = mn % g.n_tiles;
    mt = mn / g.n_tiles;
  } else {
    mt = mn % g.m_tiles;
    nt = mn / g.m_tiles;
  }
}

// ---------------------------------------------------------------------------
// tcgen05 engine
// ---------------------------------------------------------------------------
namespace tce {
constexpr int BM = 128;
constexpr int BK = 64;
constexpr int A_BYTES = BM * BK * 2;
template <int BN>
__host__ __device__ constexpr int stage_bytes() { return A_BYTES + BN * BK * 2; }
template <int BN>
__host__ __device__ constexpr uint32_t tmem_cols() {
  return (2 * BN <= 32) ? 32 : (2 * BN <= 64) ? 64 : (2 * BN <= 128) ? 128 : (2 * BN <= 256) ? 256 : 512;
}
template <int BN, int STAGES>
__host__ __device__ constexpr int smem_bytes() { return STAGES * stage_bytes<BN>() + 1024 + 512; }
}  // namespace tce

template <int BN, int STAGES, class Epi>
__global__ void __launch_bounds__(64 + 32 * EpiWarps<Epi>::value, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
                   const GemmGeom g, const __grid_constant__ Epi epi) {
  using namespace tce;
  constexpr int STAGE = stage_bytes<BN>();
  constexpr uint32_t TMEM_COLS = tmem_cols<BN>();
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "UMMA N for M=128");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* red_full = tempty + 2;
  uint64_t* red_done = red_full + 1;
  uint64_t* aux = red_done + 1;  // three one-arrival barriers the epilogue may use for its own bulk copies
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(aux + 3);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* scratch = reinterpret_cast<int*>(tmem_slot + 2);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      tc::mbar_init(full + s, 1);
      tc::mbar_init(empty + s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      tc::mbar_init(tfull + a, 1);
      tc::mbar_init(tempty + a, EpiWarps<Epi>::value);
    }
    tc::mbar_init(red_full, EpiWarps<Epi>::value * g.cluster);
    tc::mbar_init(red_done, EpiWarps<Epi>::value * g.cluster);
    for (int a = 0; a < 3; ++a) tc::mbar_init(aux + a, 1);
    *abort_flag = 0;
    tc::fence_mbar_init();
    tc::tma_prefetch_desc(&mapA);
    tc::tma_prefetch_desc(&mapB);
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, TMEM_COLS);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (g.cluster > 1) tc::cluster_sync_all();  // peers' barriers exist before any remote traffic
  const uint32_t tmem_base = *tmem_slot;
  tc::pdl_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      int last_par[STAGES];  // parity of the last load issued into each stage (-1: none)
      for (int s = 0; s < STAGES; ++s) last_par[s] = -1;
      bool ok = true;
      auto load_a = [&](uint8_t* sa, uint64_t* bar, int m0, int kb) {
        const int k0 = kb * BK;
        if (g.a3) {
          tc::tma_load_3d(sa, &mapA, bar, 0, k0, m0 / 64);
        } else if (g.a_mn) {
#pragma unroll
          for (int j = 0; j < BM / 64; ++j) tc::tma_load_2d(sa + j * 8192, &mapA, bar, m0 + 64 * j, k0);
        } else {
          tc::tma_load_2d(sa, &mapA, bar, k0, m0);
        }
      };
      auto load_b = [&](uint8_t* sb, uint64_t* bar, int n0, int kb) {
        const int k0 = kb * BK;
        if (g.b3) {
          tc::tma_load_3d(sb, &mapB, bar, 0, k0, n0 / 64);
        } else if (g.b_mn) {
#pragma unroll
          for (int j = 0; j < BN / 64; ++j) tc::tma_load_2d(sb + j * 8192, &mapB, bar, n0 + 64 * j, k0);
        } else {
          tc::tma_load_2d(sb, &mapB, bar, k0, n0);
        }
      };
      // programmatic dependent launch: the packed weights (the static operand)
      // of the first stages can stream in before the kernels this one depends
      // on finish
      int pre = 0;
      if (g.pdl) {
        if (g.static_op && (int)blockIdx.x < g.num_tiles) {
          int mt, nt, split;
          decode_tile(g, blockIdx.x, mt, nt, split);
          const int kb0 = split * g.kb_per_split;
          pre = min(STAGES, min(g.kb_total, kb0 + g.kb_per_split) - kb0);
          for (int i = 0; i < pre; ++i) {
            tc::mbar_arrive_expect_tx(full + i, STAGE);
            if (g.static_op == 1) load_a(smem + i * STAGE, full + i, mt * BM, kb0 + i);
            else load_b(smem + i * STAGE + A_BYTES, full + i, nt * BN, kb0 + i);
          }
        }
        tc::pdl_wait();
      }
      for (int tile = blockIdx.x; tile < g.num_tiles && ok; tile += gridDim.x) {
        int mt, nt, split;
        decode_tile(g, tile, mt, nt, split);
        const int kb0 = split * g.kb_per_split;
        const int kb1 = min(g.kb_total, kb0 + g.kb_per_split);
        const int m0 = mt * BM, n0 = nt * BN;
        for (int kb = kb0; kb < kb1; ++kb) {
          const bool prefilled = tile == (int)blockIdx.x && kb - kb0 < pre;  // static operand in flight, stage armed
          if (!prefilled && !tc::mbar_wait(empty + stage, phase ^ 1, abort_flag, g.err, g.limit_ns)) {
            ok = false;
            break;
          }
          uint8_t* sa = smem + stage * STAGE;
          uint8_t* sb = sa + A_BYTES;
          if (!prefilled) tc::mbar_arrive_expect_tx(full + stage, STAGE);
          last_par[stage] = static_cast<int>(phase);
          if (!prefilled || g.static_op != 1) load_a(sa, full + stage, m0, kb);
          if (!prefilled || g.static_op != 2) load_b(sb, full + stage, n0, kb);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if constexpr (EpiTail<Epi>::value) {
          if (ok && tile + (int)gridDim.x >= g.num_tiles) {
            TileCoord tt{};
            tt.m0 = m0;
            tt.n0 = n0;
            tt.mt = mt;
            tt.nt = nt;
            tt.split = split;
            tt.splits = g.splits;
            tt.cluster = g.cluster;
            tt.parts = 1;
            epi.tail_prefetch(tt, BN);
          }
        }
      }
      if (!ok) {
        // let copies already in flight land before the CTA's shared memory goes away
        for (int s = 0; s < STAGES; ++s) {
          if (last_par[s] < 0) continue;
          const uint64_t t0 = globaltimer_ns();
          while (!tc::mbar_try_wait(full + s, static_cast<uint32_t>(last_par[s])) &&
                 globaltimer_ns() - t0 < 1000000ull) {
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = tc::idesc_bf16(BM, BN, g.a_mn, g.b_mn);
      if (g.pdl) tc::pdl_wait();  // the pipeline waits below are bounded from here on
      uint32_t stage = 0, phase = 0, acc = 0, aphase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < g.num_tiles && ok; tile += gridDim.x) {
        int mt, nt, split;
        decode_tile(g, tile, mt, nt, split);
        const int kb0 = split * g.kb_per_split;
        const int kb1 = min(g.kb_total, kb0 + g.kb_per_split);
        if (!tc::mbar_wait(tempty + acc, aphase ^ 1, abort_flag, g.err, g.limit_ns)) break;
        tc::fence_after_sync();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!tc::mbar_wait(full + stage, phase, abort_flag, g.err, g.limit_ns)) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          const uint32_t sa = tc::smem_addr(smem + stage * STAGE);
          const uint32_t sb = sa + A_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t ad = g.a_mn ? tc::sdesc_sw128(sa + kk * 2048, 8192, 1024)
                                       : tc::sdesc_sw128(sa + kk * 32, 16, 1024);
            const uint64_t bd = g.b_mn ? tc::sdesc_sw128(sb + kk * 2048, 8192, 1024)
                                       : tc::sdesc_sw128(sb + kk * 32, 16, 1024);
            tc::mma_bf16(d_tmem, ad, bd, idesc, (kb > kb0 || kk > 0) ? 1u : 0u);
          }
          tc::mma_commit(empty + stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        tc::mma_commit(tfull + acc);
        acc ^= 1;
        if (acc == 0) aphase ^= 1;
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue warps
    const int q = warp & 3;  // TMEM lane quadrant this warp may access
    const int row = q * 32 + lane;
    const int part = (warp - 2) >> 2, parts = EpiWarps<Epi>::value / 4;
    if (g.pdl) tc::pdl_wait();  // the epilogue reads and writes data of earlier kernels
    uint32_t acc = 0, aphase = 0;
    const uint32_t lane_q = static_cast<uint32_t>(q * 32) << 16;
    for (int tile = blockIdx.x; tile < g.num_tiles; tile += gridDim.x) {
      int mt, nt, split;
      decode_tile(g, tile, mt, nt, split);
      const bool solo = tile == (int)blockIdx.x && tile + (int)gridDim.x >= g.num_tiles;
      typename EpiStaged<Epi>::Stash stash;
      {
        // let the epilogue's own global inputs travel to L2 (or on-chip) while the MMAs run
        TileCoord tp;
        tp.step = 0;
        tp.m0 = mt * BM;
        tp.n0 = nt * BN;
        tp.mt = mt;
        tp.nt = nt;
        tp.split = split;
        tp.splits = g.splits;
        tp.part = part;
        tp.parts = parts;
        tp.scratch = scratch;
        tp.cluster = g.cluster;
        tp.peer_base = 0;
        tp.peer_stride = 1;
        tp.red = reinterpret_cast<float*>(smem);
        tp.red_full = red_full;
        tp.red_done = red_done;
        tp.aux = aux;
        epi.prefetch(tp, row, BN);
        if constexpr (EpiStaged<Epi>::value) {
          if (solo) epi.stage(tp, row, tmem_base + BN + lane_q, BN, stash);
        }
      }
      int ok = 1;
      if (lane == 0) ok = tc::mbar_wait(tfull + acc, aphase, abort_flag, g.err, g.limit_ns) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      // every epilogue warp takes the same decision: a warp that gave up just
      // before the accumulator completed must not leave the others waiting at
      // the epilogue's named barriers
      ok = tc::bar_and(1, 32 * EpiWarps<Epi>::value, ok);
      if (!ok) break;
      tc::fence_after_sync();
      TileCoord t;
      t.step = 0;
      t.m0 = mt * BM;
      t.n0 = nt * BN;
      t.mt = mt;
      t.nt = nt;
      t.split = split;
      t.splits = g.splits;
      t.part = part;
      t.parts = parts;
      t.scratch = scratch;
      t.cluster = g.cluster;
      t.peer_base = 0;
      t.peer_stride = 1;
      t.red = reinterpret_cast<float*>(smem);
      t.red_full = red_full;
      t.red_done = red_done;
      t.aux = aux;
      TmemAcc a{tmem_base + acc * BN + lane_q};
      if constexpr (EpiStaged<Epi>::value) {
        if (solo) epi.run_staged(t, row, a, TmemAcc{tmem_base + BN + lane_q}, BN, stash);
        else epi(t, row, a, BN);
      } else {
        epi(t, row, a, BN);
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(tempty + acc);
      acc ^= 1;
      if (acc == 0) aphase ^= 1;
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem_base, TMEM_COLS);
  }
  if (g.cluster > 1) tc::cluster_sync_all();  // no peer touches this CTA's shared memory after it exits
}

// ---------------------------------------------------------------------------
// tcgen05 engine on CTA pairs (cta_group::2): a cluster of 2 CTAs computes a
// 256 x BN tile.  Each CTA loads its 128 rows of A and its BN/2 rows of B
// (so the pair reads every byte of a tile once), the even CTA issues the
// M=256 MMAs for both, each CTA's TMEM receives its 128 rows of the result
// and each CTA runs the epilogue on them.  Per SM this needs 32 KB of operand
// traffic per 64-deep K block instead of 48 KB for the same MMA work, which
// is what keeps the tensor pipe fed when the loads come from HBM.
//   full[s]    even CTA only: both CTAs' TMA bytes of stage s
//   empty[s]   both CTAs: the pair's MMAs have read stage s
//   tfull[a]   both CTAs: accumulator a is complete
//   tempty[a]  even CTA only: both CTAs' epilogues have read accumulator a
// ---------------------------------------------------------------------------
namespace tce2 {
constexpr int BM = 256;  // pair tile rows; 128 per CTA
constexpr int BK = 64;
constexpr int A_BYTES = 128 * BK * 2;
template <int BN>
__host__ __device__ constexpr int stage_bytes() { return A_BYTES + (BN / 2) * BK * 2; }
template <int BN, int STAGES>
__host__ __device__ constexpr int smem_bytes() { return STAGES * stage_bytes<BN>() + 1024 + 512; }
}  // namespace tce2

// ACCS = 2: two TMEM accumulators (the next tile's MMAs overlap this tile's
// epilogue; a CTA with a single tile stages its epilogue's inputs in the
// second).  ACCS = 1: one accumulator of BN columns and occupancy 2, for
// kernels small enough in shared memory that a second CTA (of another launch)
// shares the SM and streams its operands while this one runs its epilogue;
// two such CTAs fill the SM's 512 TMEM columns exactly.
template <int BN, int STAGES, class Epi, int ACCS = 2>
__global__ void __launch_bounds__(64 + 32 * EpiWarps<Epi>::value, ACCS == 1 ? 2 : 1)
    tc_gemm2_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
                    const GemmGeom g, const __grid_constant__ Epi epi) {
  using namespace tce2;
  constexpr int STAGE = stage_bytes<BN>();
  constexpr uint32_t TMEM_COLS = ACCS == 1 ? tce::tmem_cols<BN / 2>() : tce::tmem_cols<BN>();
  constexpr int HB = BN / 2;  // B rows per CTA
  static_assert(BN % 32 == 0 && BN >= 32 && BN <= 256, "UMMA N for M=256");
  static_assert(ACCS == 1 || ACCS == 2, "one or two accumulators");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* red_full = tempty + 2;
  uint64_t* red_done = red_full + 1;
  uint64_t* aux = red_done + 1;  // three one-arrival barriers the epilogue may use for its own bulk copies
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(aux + 3);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* scratch = reinterpret_cast<int*>(tmem_slot + 2);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // The two CTAs of a pair have cluster ranks 2i and 2i+1; the even one
  // issues the MMAs.  With split-K the cluster holds `g.cluster` such pairs.
  const uint32_t rank = tc::cluster_ctarank();
  const uint32_t leader = rank & ~1u;
  const bool is_leader = (rank & 1u) == 0;
  const uint16_t pair_mask = (uint16_t)(0x3u << leader);
  const int pr = (int)(rank & 1u);
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      tc::mbar_init(full + s, 1);
      tc::mbar_init(empty + s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      tc::mbar_init(tfull + a, 1);
      tc::mbar_init(tempty + a, 2 * EpiWarps<Epi>::value);
    }
    tc::mbar_init(red_full, EpiWarps<Epi>::value * g.cluster);
    tc::mbar_init(red_done, EpiWarps<Epi>::value * g.cluster);
    for (int a = 0; a < 3; ++a) tc::mbar_init(aux + a, 1);
    *abort_flag = 0;
    tc::fence_mbar_init();
    tc::tma_prefetch_desc(&mapA);
    tc::tma_prefetch_desc(&mapB);
  }
  if (warp == 1) {
    tc::tmem_alloc_pair(tmem_slot, TMEM_COLS);
    tc::tmem_relinquish_pair();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  tc::cluster_sync_all();  // both CTAs' barriers and TMEM exist before any pair traffic
  const uint32_t tmem_base = *tmem_slot;
  tc::pdl_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      int last_par[STAGES];
      for (int s = 0; s < STAGES; ++s) last_par[s] = -1;
      bool ok = true;
      auto load_a = [&](uint8_t* sa, uint32_t fb, int m0, int kb) {
        const int k0 = kb * BK;
        if (g.a3) {
          tc::tma_load_3d_pair(sa, &mapA, fb, 0, k0, m0 / 64);
        } else if (g.a_mn) {
#pragma unroll
          for (int j = 0; j < 2; ++j) tc::tma_load_2d_pair(sa + j * 8192, &mapA, fb, m0 + 64 * j, k0);
        } else {
          tc::tma_load_2d_pair(sa, &mapA, fb, k0, m0);
        }
      };
      auto load_b = [&](uint8_t* sb, uint32_t fb, int n0, int kb) {
        const int k0 = kb * BK;
        if (g.b3) {
          tc::tma_load_3d_pair(sb, &mapB, fb, 0, k0, n0 / 64);
        } else if (g.b_mn) {
#pragma unroll
          for (int j = 0; j < HB / 64; ++j) tc::tma_load_2d_pair(sb + j * 8192, &mapB, fb, n0 + 64 * j, k0);
        } else {
          tc::tma_load_2d_pair(sb, &mapB, fb, k0, n0);
        }
      };
      // programmatic dependent launch: the packed weights (the static operand)
      // of the first stages can stream in before the kernels this one depends
      // on finish
      int pre = 0;
      if (g.pdl) {
        if (g.static_op && pair < g.num_tiles) {
          int mt, nt, split;
          decode_tile(g, pair, mt, nt, split);
          const int kb0 = split * g.kb_per_split;
          pre = min(STAGES, min(g.kb_total, kb0 + g.kb_per_split) - kb0);
          for (int i = 0; i < pre; ++i) {
            const uint32_t fb = tc::mapa(tc::smem_addr(full + i), leader);
            if (is_leader) tc::mbar_arrive_expect_tx(full + i, 2 * STAGE);
            if (g.static_op == 1) load_a(smem + i * STAGE, fb, mt * BM + pr * 128, kb0 + i);
            else load_b(smem + i * STAGE + A_BYTES, fb, nt * BN + pr * HB, kb0 + i);
          }
        }
        tc::pdl_wait();
      }
      for (int tile = pair; tile < g.num_tiles && ok; tile += npairs) {
        int mt, nt, split, tl = tile;
        const int st_ = step_of(g, tl);
        decode_tile(g, tl, mt, nt, split);
        const int kb0 = split * g.kb_per_split;
        const int kb1 = min(g.kb_total, kb0 + g.kb_per_split);
        const int m0 = mt * BM + pr * 128, n0 = nt * BN + pr * HB + st_ * g.b_step_rows;
        int kb = kb0;
        if (st_ > 0) {
          // a later step: the stages hold this CTA's output tiles until its
          // epilogue of the step before is done, and B (h of that step) is
          // complete once every pair has stored it: one counter covers both
          if (!wait_step(g.step_cnt + st_ - 1, g.step_want, abort_flag, g.err, g.limit_ns)) {
            ok = false;
            break;
          }
          tc::fence_proxy_async_global();  // h written by other CTAs' bulk stores, read by TMA here
        }
        for (; kb < kb1; ++kb) {
          const bool prefilled = tile == pair && kb - kb0 < pre;  // static operand in flight, stage armed
          if (!prefilled && !tc::mbar_wait(empty + stage, phase ^ 1, abort_flag, g.err, g.limit_ns)) {
            ok = false;
            break;
          }
          uint8_t* sa = smem + stage * STAGE;
          uint8_t* sb = sa + A_BYTES;
          const uint32_t fb = tc::mapa(tc::smem_addr(full + stage), leader);
          if (is_leader && !prefilled) tc::mbar_arrive_expect_tx(full + stage, 2 * STAGE);
          last_par[stage] = static_cast<int>(phase);
          if (!prefilled || g.static_op != 1) load_a(sa, fb, m0, kb);
          if (!prefilled || g.static_op != 2) load_b(sb, fb, n0, kb);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (!ok && is_leader) {
        for (int s = 0; s < STAGES; ++s) {
          if (last_par[s] < 0) continue;
          const uint64_t t0 = globaltimer_ns();
          while (!tc::mbar_try_wait(full + s, static_cast<uint32_t>(last_par[s])) &&
                 globaltimer_ns() - t0 < 1000000ull) {
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (even CTA)
    if (lane == 0 && is_leader) {
      const uint32_t idesc = tc::idesc_bf16(BM, BN, g.a_mn, g.b_mn);
      if (g.pdl) tc::pdl_wait();  // the pipeline waits below are bounded from here on
      uint32_t stage = 0, phase = 0, acc = 0, aphase = 0;
      bool ok = true;
      for (int tile = pair; tile < g.num_tiles && ok; tile += npairs) {
        int mt, nt, split, tl = tile;
        step_of(g, tl);
        decode_tile(g, tl, mt, nt, split);
        const int kb0 = split * g.kb_per_split;
        const int kb1 = min(g.kb_total, kb0 + g.kb_per_split);
        if (!tc::mbar_wait(tempty + acc, aphase ^ 1, abort_flag, g.err, g.limit_ns)) break;
        tc::fence_after_sync();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!tc::mbar_wait(full + stage, phase, abort_flag, g.err, g.limit_ns)) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          const uint32_t sa = tc::smem_addr(smem + stage * STAGE);
          const uint32_t sb = sa + A_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t ad = g.a_mn ? tc::sdesc_sw128(sa + kk * 2048, 8192, 1024)
                                       : tc::sdesc_sw128(sa + kk * 32, 16, 1024);
            const uint64_t bd = g.b_mn ? tc::sdesc_sw128(sb + kk * 2048, 8192, 1024)
                                       : tc::sdesc_sw128(sb + kk * 32, 16, 1024);
            tc::mma_bf16_pair(d_tmem, ad, bd, idesc, (kb > kb0 || kk > 0) ? 1u : 0u);
          }
          tc::mma_commit_pair(empty + stage, pair_mask);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        tc::mma_commit_pair(tfull + acc, pair_mask);
        if (ACCS == 2) acc ^= 1;
        if (acc == 0) aphase ^= 1;
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue warps (both CTAs)
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const int part = (warp - 2) >> 2, parts = EpiWarps<Epi>::value / 4;
    const uint32_t te_base = tc::mapa(tc::smem_addr(tempty), leader);
    if (g.pdl) tc::pdl_wait();  // the epilogue reads and writes data of earlier kernels
    uint32_t acc = 0, aphase = 0;
    const uint32_t lane_q = static_cast<uint32_t>(q * 32) << 16;
    for (int tile = pair; tile < g.num_tiles; tile += npairs) {
      int mt, nt, split, tl = tile;
      const int st_ = step_of(g, tl);
      decode_tile(g, tl, mt, nt, split);
      // a CTA with one tile stages its epilogue inputs in the idle second
      // accumulator; over several dependent steps, in the accumulator of the
      // step before (its epilogue is done, and the next step's products wait
      // for this step's stores in every CTA)
      const bool solo = (tile == pair && tile + npairs >= g.num_tiles) || g.steps > 1;
      const uint32_t st_col = (acc ^ 1u) * BN;
      typename EpiStaged<Epi>::Stash stash;
      TileCoord t;
      t.step = st_;
      t.m0 = mt * BM + pr * 128;
      t.n0 = nt * BN;
      t.mt = mt * 2 + pr;
      t.nt = nt;
      t.split = split;
      t.splits = g.splits;
      t.part = part;
      t.parts = parts;
      t.scratch = scratch;
      t.cluster = g.cluster;  // > 1: the splits reduce through the cluster, pairs interleaved
      t.peer_base = pr;
      t.peer_stride = 2;
      t.red = reinterpret_cast<float*>(smem);
      t.red_full = red_full;
      t.red_done = red_done;
      t.aux = aux;
      epi.prefetch(t, row, BN);
      if constexpr (EpiStaged<Epi>::value && ACCS == 2) {
        if (solo) epi.stage(t, row, tmem_base + st_col + lane_q, BN, stash);
      }
      int ok = 1;
      if (lane == 0) ok = tc::mbar_wait(tfull + acc, aphase, abort_flag, g.err, g.limit_ns) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      // every epilogue warp takes the same decision: a warp that gave up just
      // before the accumulator completed must not leave the others waiting at
      // the epilogue's named barriers
      ok = tc::bar_and(1, 32 * EpiWarps<Epi>::value, ok);
      if (!ok) break;
      tc::fence_after_sync();
      TmemAcc a{tmem_base + acc * BN + lane_q};
      if constexpr (EpiStaged<Epi>::value && ACCS == 2) {
        if (solo) epi.run_staged(t, row, a, TmemAcc{tmem_base + st_col + lane_q}, BN, stash);
        else epi(t, row, a, BN);
      } else {
        epi(t, row, a, BN);
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive_remote(te_base + acc * 8);
      if (ACCS == 2) acc ^= 1;
      if (acc == 0) aphase ^= 1;
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  tc::cluster_sync_all();  // the pair's MMAs and remote arrivals are done before TMEM and smem go away
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// fp32 SIMT engine (FFMA): 32 x BN tiles, 128 threads, K step 16.
//
// Every dot product is accumulated with compensation: the "Dot2" scheme of
// Ogita, Rump and Oishi ("Accurate sum and dot product", SIAM J. Sci. Comput.
// 26(6), 2005).  Each product a*b is split exactly into p + pe with one FMA
// (pe = fma(a, b, -p)), p is added to the running sum by Knuth's TwoSum, which
// also yields the exact rounding error of that addition, and both errors are
// collected in a second float.  The result is as accurate as a sum taken in
// twice the working precision and rounded once, whatever K is; a plain
// sequential fp32 sum instead carries an error that grows with K and, where
// an output is a small difference of O(1) terms, exceeds the fp32 mode's
// 1e-4 relative bound.  All operations are fp32 (no TF32, no fp64); the
// explicit _rn intrinsics keep the compiler from contracting or reordering
// them.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void dot2_add(float a, float b, float& hi, float& lo) {
  const float p = __fmul_rn(a, b);
  const float pe = __fmaf_rn(a, b, -p);  // a*b - p, exactly
  const float s = __fadd_rn(hi, p);
  const float bv = __fsub_rn(s, hi);
  const float e = __fadd_rn(__fsub_rn(hi, __fsub_rn(s, bv)), __fsub_rn(p, bv));  // hi + p - s, exactly
  hi = s;
  lo = __fadd_rn(lo, __fadd_rn(e, pe));
}
// Compensated sum of floats (the same TwoSum step without the product).
__device__ __forceinline__ void sum2_add(float v, float& hi, float& lo) {
  const float s = __fadd_rn(hi, v);
  const float bv = __fsub_rn(s, hi);
  lo = __fadd_rn(lo, __fadd_rn(__fsub_rn(hi, __fsub_rn(s, bv)), __fsub_rn(v, bv)));
  hi = s;
}

namespace se {
constexpr int BM = 32;
constexpr int BK = 16;
template <int BN>
__host__ __device__ constexpr int smem_bytes() { return (BK * (BM + 1) + BK * (BN + 1) + BM * (BN + 1)) * 4; }
}  // namespace se

template <int BN, class Epi>
__global__ void __launch_bounds__(128)
    simt_gemm_kernel(const float* __restrict__ A, long long lda, const float* __restrict__ Bm, long long ldb,
                     const GemmGeom g, const Epi epi) {
  using namespace se;
  static_assert(BN % 32 == 0, "SIMT tile width");
  constexpr int NC = BN / 32;
  extern __shared__ float sm[];
  float* As = sm;                          // [BK][BM+1]
  float* Bs = As + BK * (BM + 1);          // [BK][BN+1]
  float* Cs = Bs + BK * (BN + 1);          // [BM][BN+1]
  const int tid = threadIdx.x;
  const int ty = tid >> 5, tx = tid & 31;
  int mt, nt, split;
  decode_tile(g, blockIdx.x, mt, nt, split);
  const int m0 = mt * BM, n0 = nt * BN;
  float acc[8][NC], err[8][NC];  // compensated sums: value and collected rounding errors
#pragma unroll
  for (int r = 0; r < 8; ++r)
#pragma unroll
    for (int c = 0; c < NC; ++c) acc[r][c] = err[r][c] = 0.f;

  for (int k0 = 0; k0 < g.K; k0 += BK) {
    for (int e = tid; e < BM * BK; e += 128) {
      const int r = e / BK, kk = e % BK;
      const int m = m0 + r, k = k0 + kk;
      float v = 0.f;
      if (m < g.M && k < g.K) v = g.a_mn ? A[(long long)k * lda + m] : A[(long long)m * lda + k];
      As[kk * (BM + 1) + r] = v;
    }
    for (int e = tid; e < BN * BK; e += 128) {
      const int c = e / BK, kk = e % BK;
      const int n = n0 + c, k = k0 + kk;
      float v = 0.f;
      if (n < g.N && k < g.K) v = g.b_mn ? Bm[(long long)k * ldb + n] : Bm[(long long)n * ldb + k];
      Bs[kk * (BN + 1) + c] = v;
    }
    __syncthreads();
#pragma unroll 4
    for (int kk = 0; kk < BK; ++kk) {
      float a[8], b[NC];
#pragma unroll
      for (int r = 0; r < 8; ++r) a[r] = As[kk * (BM + 1) + ty * 8 + r];
#pragma unroll
      for (int c = 0; c < NC; ++c) b[c] = Bs[kk * (BN + 1) + tx + 32 * c];
#pragma unroll
      for (int r = 0; r < 8; ++r)
#pragma unroll
        for (int c = 0; c < NC; ++c) dot2_add(a[r], b[c], acc[r][c], err[r][c]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int r = 0; r < 8; ++r)
#pragma unroll
    for (int c = 0; c < NC; ++c) Cs[(ty * 8 + r) * (BN + 1) + tx + 32 * c] = __fadd_rn(acc[r][c], err[r][c]);
  __syncthreads();
  // one thread per tile row, or EpiSimtShares of them sharing out its
  // elements; with few rows in the tile (a small batch) the shares double
  // while the block has threads for them, up to 32 per row
  constexpr int ES = EpiSimtShares<Epi>::value;
  static_assert(ES * BM <= 128, "shares of a tile row");
  const int nrow = ES > 1 ? max(1, min(BM, g.M - m0)) : BM;
  int es = ES;
  if (ES > 1)
    while (es < 32 && 2 * es * nrow <= 128) es *= 2;
  if (tid < es * nrow) {
    const int row = tid % nrow;
    TileCoord t;
    t.step = 0;
    t.part = tid / nrow;
    t.parts = es;
    t.m0 = m0;
    t.n0 = n0;
    t.mt = mt;
    t.nt = nt;
    t.split = 0;
    t.splits = 1;
    t.scratch = nullptr;
    t.cluster = 1;
    t.peer_base = 0;
    t.peer_stride = 1;
    t.red = nullptr;
    t.red_full = t.red_done = nullptr;
    SmemAcc a{Cs + row * (BN + 1)};
    epi(t, row, a, BN);
  }
}

}  // namespace rnn
