// stack.cu -- persistent forward recurrence of a group of stacked layers for
// moderate batches (9 to 64 sequences), all timesteps in one launch.
//
// "Persistent RNNs: Stashing Recurrent Weights On-Chip" (citing snippets on
// its page): keep the recurrent weights on chip across timesteps and run the
// whole sequence in one kernel launch.  "Optimizing Performance of RNNs on
// GPUs" (review page, proposed method): the layers of a stack overlap in a
// wavefront, layer l working on step t while layer l+1 works on step t-1.
// Here both happen inside one launch:
//
//  * Every layer of the group owns its CTAs.  A CTA holds one block of 128
//    packed gate rows (all gates of 32 hidden units; 128 units for the
//    simple RNNs) times one 512-wide (or 256-wide) chunk of the layer's K =
//    [input | recurrent] in shared memory for the whole launch, in the
//    tensor core's 128-byte-swizzled K-major layout.  The first layer of the
//    whole stack takes its input projection P = x W_x^T + b from one GEMM
//    over all timesteps and its K is the recurrent part only; every other
//    layer computes its input projection step by step from the layer
//    below's h_t (the K chunks of the input part), so a layer can start step
//    t as soon as the layer below has finished it.
//  * Per timestep a CTA waits for the arrival counter of what its chunk
//    reads (the layer below's step t for an input chunk, its own layer's
//    step t-1 for a recurrent chunk), then one thread streams the batch rows
//    of that chunk (N = batch rounded up to 16, x 64 k per block) from L2
//    into a ring of shared-memory stages with TMA, and one thread issues
//    tcgen05.mma (M = 128 rows, N, K = 16) into a double-buffered TMEM
//    accumulator.
//  * The K chunks of one row block form a thread-block cluster.  Their
//    partial sums are reduce-scattered over the batch: each CTA sends the
//    other chunks' batch slices with asynchronous stores into their shared
//    memory (counted on their mbarriers) and adds the slices it receives to
//    its own in chunk order (deterministic).  Each CTA then owns all G gate
//    rows of its 32 units for its slice of the batch: it adds the bias (or
//    P), applies the activations and the cell update (c and, for GRU,
//    h_{t-1} stay in registers across steps), writes h_t (bf16), the
//    activated gates and c (training) and makes one release arrival on its
//    layer's counter of step t.
//
// GRU keeps the input and recurrent parts of the candidate gate apart (the
// reset gate multiplies only the recurrent part): its chunks are each purely
// input or purely recurrent, and the reduction sums the two kinds apart.
//
// Every wait is bounded (globaltimer).  A CTA that gives up records
// DEV_TIMEOUT_STEP / DEV_TIMEOUT_PIPE in the error word, marks the abort
// flag of every CTA of its cluster and leaves its loop; in-flight copies and
// MMAs are waited for (bounded) before the CTA frees its tensor memory, and a
// final cluster barrier keeps every CTA resident until no peer can still
// store into its shared memory.  All CTAs are co-resident (cooperative
// launch), so the counters a CTA waits for are always being worked on.
#include <cuda.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <cstring>

#include "../../include/rnn.h"
#include "common.cuh"
#include "launch.cuh"
#include "launchers.h"
#include "tc.cuh"

namespace rnn {

namespace {

#define RNN_TRY_LOCAL(x)          \
  do {                            \
    const int rc_ = (x);          \
    if (rc_ != RNN_OK) return rc_; \
  } while (0)

// TMA maps of one launch: packed W_x and W_h rows of each layer (box 64 k x
// 128 rows) and the h sequences (box 64 k x N batch rows): h[0] the input
// of the first layer (when it has no P), h[1 + l] layer l's own.
struct StackMaps {
  CUtensorMap wx[kStackMaxLayers];
  CUtensorMap wh[kStackMaxLayers];
  CUtensorMap h[kStackMaxLayers + 1];
};

constexpr int kStages = 4;
constexpr int kThreads = 192;  // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue (one per TMEM lane quadrant)

__device__ __forceinline__ unsigned int ld_acquire_u32(const unsigned int* p) {
  unsigned int v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void red_release_add_u32(unsigned int* p, unsigned int v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void st_async_v4(uint32_t cluster_addr, const float* v, uint32_t cluster_bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
                   cluster_addr),
               "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
               "r"(__float_as_uint(v[3])), "r"(cluster_bar)
               : "memory");
}
__device__ __forceinline__ void st_dsmem_s32(uint32_t cluster_addr, int v) {
  asm volatile("st.shared::cluster.s32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}

// Shared-memory layout of a CTA (offsets from the 1024-aligned base).
struct Smem {
  int a, ring, rbuf, smg, smhn, bars, total;
};
__host__ __device__ inline Smem smem_layout(int cell, int N, int kc, int ksmin, int ksmax) {
  Smem s;
  s.a = 0;
  s.ring = s.a + (kc / 64) * 16384;
  s.rbuf = s.ring + kStages * N * 128;
  // [2][ksmax-1][N/ks/4][128] float4 for the largest ks of the launch (the
  // footprint (ks-1)/ks * N is largest for the largest ks)
  const int rb = ksmax > 1 ? 2 * (ksmax - 1) * (N / ksmax) * 128 * 4 : 0;
  s.smg = s.rbuf + rb;
  // gate tile [N/ks][128] and GRU recurrent candidate part [N/ks][32] for the
  // widest batch slice of the launch (smallest ks)
  s.smhn = s.smg + (N / ksmin) * 128 * 4;
  s.bars = s.smhn + (cell == GRU ? (N / ksmin) * 32 * 4 : 0);
  s.total = s.bars + 256;
  return s;
}

struct Ctx {
  uint8_t* smem;
  uint64_t *full, *empty, *tfull, *tempty, *rbar, *abar, *dbar;
  uint32_t tmem;
  volatile int* abort_flag;
  int* ep_fail;
  int li, rb, me, ks, kcx, crank;
};

// Raise the abort flag in every CTA of the cluster (this one included).
__device__ __forceinline__ void abort_cluster(const Ctx& c, int cluster) {
  *c.abort_flag = 1;
  if (cluster > 1) {
    const uint32_t fa = tc::smem_addr(const_cast<int*>(c.abort_flag));
    for (int r = 0; r < cluster; ++r) st_dsmem_s32(tc::mapa(fa, (uint32_t)r), 1);
  }
}

// Wait until *cnt >= want (bounded; gives up at once when the CTA aborts).
__device__ __forceinline__ bool wait_count(const unsigned int* cnt, unsigned int want, const Ctx& c,
                                           const StackArgs& a) {
  if (ld_acquire_u32(cnt) >= want) return true;
  const uint64_t t0 = globaltimer_ns();
  while (ld_acquire_u32(cnt) < want) {
    if (*c.abort_flag) return false;
    if (globaltimer_ns() - t0 > a.limit_ns) {
      raise_error(a.err, DEV_TIMEOUT_STEP);
      abort_cluster(c, a.cluster);
      return false;
    }
  }
  return true;
}

// ---------------------------------------------------------------------------
// epilogue: 128 threads, thread e owns TMEM lane / packed row `row` of the
// CTA's block; KS chunks per row block, this CTA's batch slice is
// [me*NS, me*NS + NS)
template <int CELL, int N, int KS>
__device__ void epilogue(const StackArgs& a, const Ctx& c, int row, int e) {
  constexpr int G = CellInfo<CELL>::G;
  constexpr bool SIMPLE = G == 1;
  constexpr int UC = SIMPLE ? 128 : 32;
  constexpr int ROWS = G * UC;
  constexpr int NS = N / KS;
  constexpr int PP = SIMPLE ? 1 : (UC * NS + 127) / 128;  // (unit, batch) pairs per thread
  const StackLayer& ly = a.lay[c.li];
  const int T = a.T, B = a.B, H = a.H, GH = G * H, u = a.u_pack;
  const int me = c.me, kcx = c.kcx;
  const int j0 = c.rb * UC, r0 = j0 * G;
  const int lane = threadIdx.x & 31;
  const uint32_t lane_q = static_cast<uint32_t>(row & ~31) << 16;
  const bool live_row = row < ROWS;
  // gate and unit of this thread's row
  const int rg = (row % (G * u)) / u;
  const int rj = (row / (G * u)) * u + row % u;
  const float bias = (live_row && !ly.P) ? ly.bias[r0 + row] : 0.f;
  const float bias_hn = (CELL == GRU && live_row && rg == 2) ? ly.bias_hn[j0 + rj] : 0.f;
  float* smg = reinterpret_cast<float*>(c.smem + a.sm.smg);
  float* smhn = reinterpret_cast<float*>(c.smem + a.sm.smhn);
  float4* rbuf = reinterpret_cast<float4*>(c.smem + a.sm.rbuf);
  constexpr int NC4 = NS / 4;  // float4 chunks of a slice
  constexpr int ACC = N < 32 ? 32 : N;  // TMEM columns between the two accumulators
  // receive buffer of parity p from the peer in slot s: [p][s][chunk][row]
  auto rb_at = [&](int p, int s, int ch) -> float4* { return rbuf + ((p * (KS - 1) + s) * NC4 + ch) * 128; };

  // per-pair state (LSTM c, GRU h_{t-1}) kept across steps
  float st[PP];
#pragma unroll
  for (int i = 0; i < PP; ++i) {
    st[i] = 0.f;
    if constexpr (!SIMPLE) {
      const int q = i * 128 + e, jl = q % UC, cc = q / UC, b = me * NS + cc;
      if (cc < NS && b < B) {
        if (CELL == LSTM && ly.c0) st[i] = ly.c0[(size_t)b * H + j0 + jl];
        if (CELL == GRU) st[i] = __bfloat162float(ly.hseq[(size_t)b * H + j0 + jl]);
      }
    }
  }

  for (int t = 0; t < T; ++t) {
    const int acc = t & 1, par = t & 1;
    const uint32_t ph = (uint32_t)(t >> 1) & 1u;
    if (KS > 1 && e == 0) tc::mbar_arrive_expect_tx(&c.rbar[par], (uint32_t)((KS - 1) * 128 * NS * 4));
    // sx: input part (the first layer's input projection P, loaded before the
    // accumulator is ready, or the folded bias plus the input chunks); sh:
    // recurrent part (GRU only: the other cells add everything into sx)
    constexpr bool SPLIT = CELL == GRU;
    float sx[NS], sh[SPLIT ? NS : 1];
#pragma unroll
    for (int cc = 0; cc < NS; ++cc) {
      const int b = me * NS + cc;
      sx[cc] = ly.P ? ((live_row && b < B) ? ly.P[((size_t)t * B + b) * GH + r0 + row] : 0.f) : bias;
      if constexpr (SPLIT) sh[cc] = 0.f;
    }
    // ---- accumulator of this step
    bool ok = true;
    {
      int w = 1;
      if (lane == 0) w = tc::mbar_wait(&c.tfull[acc], ph, c.abort_flag, a.err, a.limit_ns) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, w, 0) != 0;
    }
    if (ok) {
      tc::fence_after_sync();
      // the accumulator 16 columns at a time: each group of 4 columns is either
      // this CTA's batch slice (added to its sums) or another chunk's (sent
      // into that CTA's receive buffer)
#pragma unroll
      for (int i = 0; i < N / 16; ++i) {
        float w[16];
        tc::tmem_load16(c.tmem + lane_q + (uint32_t)(acc * ACC + 16 * i), w);
#pragma unroll
        for (int g4 = 0; g4 < 4; ++g4) {
          const int col = 16 * i + 4 * g4, p = col / NS, cc = col % NS;
          if (p == me) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              if (SPLIT && me >= kcx) sh[cc + q] += w[4 * g4 + q];
              else sx[cc + q] += w[4 * g4 + q];
            }
          } else if constexpr (KS > 1) {
            const int slot = me < p ? me : me - 1;
            const uint32_t prank = (uint32_t)(c.crank - me + p);
            st_async_v4(tc::mapa(tc::smem_addr(rb_at(par, slot, cc / 4) + row), prank), w + 4 * g4,
                        tc::mapa(tc::smem_addr(&c.rbar[par]), prank));
          }
        }
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&c.tempty[acc]);
      if constexpr (KS > 1) {
        int w = 1;
        if (lane == 0) {
          w = 0;
          const uint64_t t0 = globaltimer_ns();
          while (true) {
            if (tc::mbar_try_wait_cluster(&c.rbar[par], ph)) {
              w = 1;
              break;
            }
            if (*c.abort_flag) break;
            if (globaltimer_ns() - t0 > a.limit_ns) {
              raise_error(a.err, DEV_TIMEOUT_STEP);
              break;
            }
          }
        }
        ok = __shfl_sync(0xffffffffu, w, 0) != 0;
      }
    }
    if (!ok && lane == 0) {
      *c.ep_fail = 1;
      abort_cluster(c, a.cluster);
    }
    tc::named_bar(1, 128);
    if (*reinterpret_cast<volatile int*>(c.ep_fail)) break;

    // ---- the other chunks' partial sums of this CTA's slice, in chunk order
    // (input and recurrent parts apart for GRU)
#pragma unroll
    for (int k = 0; k < KS; ++k) {
      if (k == me) continue;
      const bool xk = !SPLIT || k < kcx;
      const int slot = k < me ? k : k - 1;
#pragma unroll
      for (int ch = 0; ch < NC4; ++ch) {
        const float4 q = rb_at(par, slot, ch)[row];
        const float qq[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          if (SPLIT && !xk) sh[4 * ch + i] += qq[i];
          else sx[4 * ch + i] += qq[i];
        }
      }
    }

    // ---- gates of this row for the batch slice
    const size_t tb = (size_t)t * B;
#pragma unroll
    for (int cc = 0; cc < NS; ++cc) {
      const int b = me * NS + cc;
      if (!live_row || b >= B) continue;
      if constexpr (CELL == LSTM) {
        const float pre = sx[cc];
        const float gv = rg == 2 ? tanh_hw(pre) : sigm_hw(pre);
        if (ly.gates_out) ly.gates_out[(tb + b) * GH + r0 + row] = gv;
        smg[cc * 128 + row] = gv;
      } else if constexpr (CELL == GRU) {
        if (rg < 2) {
          const float gv = sigm_hw(sx[cc] + sh[cc]);
          if (ly.gates_out) ly.gates_out[(tb + b) * GH + r0 + row] = gv;
          smg[cc * 128 + row] = gv;
        } else {
          smg[cc * 128 + row] = sx[cc];           // x_n + b_xn
          smhn[cc * 32 + rj] = sh[cc] + bias_hn;  // W_hn h_{t-1} + b_hn
        }
      } else {
        const float hv = simple_act<CELL, __nv_bfloat16>(sx[cc]);
        const __nv_bfloat16 hb = __float2bfloat16_rn(hv);
        const size_t bj = (size_t)b * H + j0 + row;
        if (ly.gates_out) ly.gates_out[(tb + b) * GH + r0 + row] = hv;
        ly.hseq[(size_t)(t + 1) * B * H + bj] = hb;
        if (ly.y) ly.y[tb * H + bj] = hb;
        if (t == T - 1 && ly.hT) ly.hT[bj] = hb;
      }
    }
    if constexpr (!SIMPLE) {
      tc::named_bar(1, 128);
      // ---- cell update of this thread's (unit, batch entry) pairs
#pragma unroll
      for (int i = 0; i < PP; ++i) {
        const int q = i * 128 + e, jl = q % UC, cc = q / UC, b = me * NS + cc;
        if (cc >= NS || b >= B) continue;
        const int j = j0 + jl;
        const size_t bj = (size_t)b * H + j;
        const float* gr = smg + cc * 128;
        float hv;
        if constexpr (CELL == LSTM) {
          float ig, fg, gg, og;
          if (u == 1) {
            const float4 g4 = *reinterpret_cast<const float4*>(gr + 4 * jl);
            ig = g4.x; fg = g4.y; gg = g4.z; og = g4.w;
          } else {
            ig = gr[packed_row(0, jl, 4, u)];
            fg = gr[packed_row(1, jl, 4, u)];
            gg = gr[packed_row(2, jl, 4, u)];
            og = gr[packed_row(3, jl, 4, u)];
          }
          st[i] = fg * st[i] + ig * gg;
          hv = og * tanh_hw(st[i]);
          if (ly.c_out) ly.c_out[tb * H + bj] = st[i];
          if (t == T - 1 && ly.cT) ly.cT[bj] = st[i];
        } else {
          const float r = gr[packed_row(0, jl, 3, u)], z = gr[packed_row(1, jl, 3, u)];
          const float xn = gr[packed_row(2, jl, 3, u)], hn = smhn[cc * 32 + jl];
          const float n = tanh_hw(xn + r * hn);
          hv = (1.f - z) * n + z * st[i];
          st[i] = hv;
          if (ly.gates_out) ly.gates_out[(tb + b) * GH + r0 + packed_row(2, jl, 3, u)] = n;
          if (ly.hn_out) ly.hn_out[tb * H + bj] = hn;
        }
        const __nv_bfloat16 hb = __float2bfloat16_rn(hv);
        ly.hseq[(size_t)(t + 1) * B * H + bj] = hb;
        if (ly.y) ly.y[tb * H + bj] = hb;
        if (t == T - 1 && ly.hT) ly.hT[bj] = hb;
      }
    }
    // ---- publish h_t of this CTA's units and batch slice: the readers load
    // it with TMA (async proxy) after acquiring the counter
    tc::fence_proxy_async_global();
    tc::named_bar(1, 128);
    if (e == 0 && !(a.test_skip_publish && blockIdx.x == 0 && t == 0))
      red_release_add_u32(a.cnt + (size_t)c.li * T + t, 1u);
  }
}

template <int CELL, int N>
__global__ void __launch_bounds__(kThreads, 1)
    stack_fwd_kernel(const __grid_constant__ StackMaps maps, const StackArgs a) {
  constexpr int G = CellInfo<CELL>::G;
  constexpr int UC = G == 1 ? 128 : 32;
  constexpr int RING = N * 128;
  constexpr int ACC = N < 32 ? 32 : N;  // TMEM columns between the two accumulators
  constexpr uint32_t TMEM_COLS = 2 * ACC <= 64 ? 64 : 128;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (a.cluster > 1) {
    uint32_t ncta;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(ncta));
    if ((int)ncta != a.cluster) {
      if (threadIdx.x == 0) raise_error(a.err, DEV_BAD_CLUSTER);
      return;
    }
  }
  Ctx c;
  c.smem = smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + a.sm.bars);
  c.full = bars;
  c.empty = c.full + kStages;
  c.tfull = c.empty + kStages;
  c.tempty = c.tfull + 2;
  c.rbar = c.tempty + 2;
  c.abar = c.rbar + 2;
  c.dbar = c.abar + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(c.dbar + 1);
  c.abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  c.ep_fail = reinterpret_cast<int*>(tmem_slot + 2);
  c.li = 0;
  while (c.li + 1 < a.nl && (int)blockIdx.x >= a.cta0[c.li + 1]) ++c.li;
  c.ks = a.ks[c.li];
  c.kcx = a.kcx[c.li];
  const int local = (int)blockIdx.x - a.cta0[c.li];
  c.rb = local / c.ks;
  c.me = local % c.ks;
  c.crank = a.cluster > 1 ? (int)tc::cluster_ctarank() : 0;
  const StackLayer& ly = a.lay[c.li];
  const bool xpart = c.me < c.kcx;
  const int k0 = (xpart ? c.me : c.me - c.kcx) * a.kc;
  const int nkb = a.kc / 64;
  const int r0 = c.rb * UC * G;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      tc::mbar_init(c.full + s, 1);
      tc::mbar_init(c.empty + s, 1);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(c.tfull + i, 1);
      tc::mbar_init(c.tempty + i, 4);
      tc::mbar_init(c.rbar + i, 1);
    }
    tc::mbar_init(c.abar, 1);
    tc::mbar_init(c.dbar, 1);
    *c.abort_flag = 0;
    *c.ep_fail = 0;
    tc::fence_mbar_init();
    tc::tma_prefetch_desc(xpart ? &maps.wx[c.li] : &maps.wh[c.li]);
    tc::tma_prefetch_desc(xpart ? &maps.h[c.li] : &maps.h[c.li + 1]);
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, TMEM_COLS);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (a.cluster > 1) tc::cluster_sync_all();  // every peer's barriers and flags exist before remote traffic
  c.tmem = *tmem_slot;

  int last_par[kStages];  // producer: parity of the last load issued into each stage (-1: none)
  for (int s = 0; s < kStages; ++s) last_par[s] = -1;
  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      // this CTA's block of weight rows, resident for the whole launch
      tc::mbar_arrive_expect_tx(c.abar, (uint32_t)nkb * 16384u);
      for (int kb = 0; kb < nkb; ++kb)
        tc::tma_load_2d(smem + a.sm.a + kb * 16384, xpart ? &maps.wx[c.li] : &maps.wh[c.li], c.abar, k0 + kb * 64,
                        r0);
      uint32_t stage = 0, phase = 0;
      const CUtensorMap* src = xpart ? &maps.h[c.li] : &maps.h[c.li + 1];
      for (int t = 0; t < a.T; ++t) {
        bool ok = true;
        if (xpart) {
          if (ly.wait_in) ok = wait_count(a.cnt + (size_t)(c.li - 1) * a.T + t, (unsigned)a.ctas[c.li - 1], c, a);
        } else if (t > 0) {
          ok = wait_count(a.cnt + (size_t)c.li * a.T + t - 1, (unsigned)a.ctas[c.li], c, a);
        }
        if (!ok) break;
        // h written by other CTAs' generic stores, read here through the async proxy
        tc::fence_proxy_async_global();
        const int slot = xpart ? t + 1 : t;
        for (int kb = 0; kb < nkb && ok; ++kb) {
          if (!tc::mbar_wait(c.empty + stage, phase ^ 1, c.abort_flag, a.err, a.limit_ns)) {
            ok = false;
            break;
          }
          tc::mbar_arrive_expect_tx(c.full + stage, RING);
          last_par[stage] = (int)phase;
          tc::tma_load_2d(smem + a.sm.ring + stage * RING, src, c.full + stage, k0 + kb * 64, slot * a.B);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
      }
      if (*c.abort_flag) abort_cluster(c, a.cluster);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = tc::idesc_bf16(128, N, 0, 0);
      bool ok = tc::mbar_wait(c.abar, 0, c.abort_flag, a.err, a.limit_ns);
      tc::fence_after_sync();
      uint32_t stage = 0, phase = 0;
      const uint32_t sa = tc::smem_addr(smem + a.sm.a);
      for (int t = 0; t < a.T && ok; ++t) {
        const int acc = t & 1;
        if (!tc::mbar_wait(c.tempty + acc, ((uint32_t)(t >> 1) & 1u) ^ 1u, c.abort_flag, a.err, a.limit_ns)) break;
        tc::fence_after_sync();
        const uint32_t d = c.tmem + (uint32_t)(acc * ACC);
        for (int kb = 0; kb < nkb; ++kb) {
          if (!tc::mbar_wait(c.full + stage, phase, c.abort_flag, a.err, a.limit_ns)) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          const uint32_t sb = tc::smem_addr(smem + a.sm.ring + stage * RING);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            tc::mma_bf16(d, tc::sdesc_sw128(sa + kb * 16384 + kk * 32, 16, 1024),
                         tc::sdesc_sw128(sb + kk * 32, 16, 1024), idesc, (kb > 0 || kk > 0) ? 1u : 0u);
          tc::mma_commit(c.empty + stage);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        tc::mma_commit(c.tfull + acc);
      }
      // every MMA issued has completed before the tensor memory is freed
      tc::mma_commit(c.dbar);
      const uint64_t t0 = globaltimer_ns();
      while (!tc::mbar_try_wait(c.dbar, 0) && globaltimer_ns() - t0 < 1000000ull) {
      }
      if (*c.abort_flag) abort_cluster(c, a.cluster);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int row = (warp & 3) * 32 + lane;
    const int e = threadIdx.x - 64;
    if (c.ks == 1) epilogue<CELL, N, 1>(a, c, row, e);
    else if (c.ks == 2) epilogue<CELL, N, 2>(a, c, row, e);
    else epilogue<CELL, N, 4>(a, c, row, e);
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0 && lane == 0 && *c.abort_flag) {
    // copies already issued land before the CTA's shared memory goes away
    // (after an abort some were never consumed)
    for (int s = 0; s < kStages; ++s) {
      if (last_par[s] < 0) continue;
      const uint64_t t0 = globaltimer_ns();
      while (!tc::mbar_try_wait(c.full + s, (uint32_t)last_par[s]) && globaltimer_ns() - t0 < 1000000ull) {
      }
    }
    const uint64_t t0 = globaltimer_ns();
    while (!tc::mbar_try_wait(c.abar, 0) && globaltimer_ns() - t0 < 1000000ull) {
    }
  }
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(c.tmem, TMEM_COLS);
  }
  if (a.cluster > 1) tc::cluster_sync_all();  // no peer stores into this CTA's shared memory after it exits
}

// Geometry of a launch over layers [0, nl) of a group: K chunk, chunks per
// layer, CTAs.  first_p: the group's first layer reads P (it is the stack's
// layer 0).
struct Geom {
  int kc, N, cluster, ctas;
  int ks[kStackMaxLayers], kcx[kStackMaxLayers], cta0[kStackMaxLayers + 1], lctas[kStackMaxLayers];
  Smem sm;
};

int geometry(int cell, int H, int B, int nl, int first_p, Geom* g) {
  if (nl < 1 || nl > kStackMaxLayers || B < 1 || B > 64) return RNN_ERR_UNSUPPORTED;
  const int G = cell == LSTM ? 4 : cell == GRU ? 3 : 1;
  const int uc = G == 1 ? 128 : 32;
  if (H % uc) return RNN_ERR_UNSUPPORTED;
  g->kc = H % 512 == 0 ? 512 : H % 256 == 0 ? 256 : 0;
  if (!g->kc) return RNN_ERR_UNSUPPORTED;
  g->N = B <= 16 ? 16 : B <= 32 ? 32 : 64;
  const int rbs = H / uc;
  int cta = 0, ksmax = 1, ksmin = 4;
  for (int l = 0; l < nl; ++l) {
    const bool p = l == 0 && first_p;
    g->kcx[l] = p ? 0 : H / g->kc;  // layers above the first: input width H
    g->ks[l] = g->kcx[l] + H / g->kc;
    if (g->ks[l] != 1 && g->ks[l] != 2 && g->ks[l] != 4) return RNN_ERR_UNSUPPORTED;
    if (g->N / g->ks[l] < 4) return RNN_ERR_UNSUPPORTED;
    ksmax = std::max(ksmax, g->ks[l]);
    ksmin = std::min(ksmin, g->ks[l]);
    g->cta0[l] = cta;
    g->lctas[l] = rbs * g->ks[l];
    cta += g->lctas[l];
  }
  g->cta0[nl] = cta;
  g->ctas = cta;
  g->cluster = ksmax;
  for (int l = 0; l < nl; ++l)
    if (g->lctas[l] % ksmax) return RNN_ERR_UNSUPPORTED;
  g->sm = smem_layout(cell, g->N, g->kc, ksmin, ksmax);
  if (g->sm.total + 1024 > 227 * 1024) return RNN_ERR_UNSUPPORTED;
  return RNN_OK;
}

template <int CELL, int N>
int launch_t(const Launch& L, const StackMaps& maps, const StackArgs& a, const Geom& g, bool query_only,
             int num_sms) {
  auto k = stack_fwd_kernel<CELL, N>;
  const int dyn = g.sm.total + 1024;
  if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn) != cudaSuccess) {
    (void)cudaGetLastError();
    return RNN_ERR_UNSUPPORTED;
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(g.ctas);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = dyn;
  cfg.stream = L.stream;
  cudaLaunchAttribute at[2];
  unsigned n = 0;
  if (g.cluster > 1) {
    at[n].id = cudaLaunchAttributeClusterDimension;
    at[n].val.clusterDim.x = g.cluster;
    at[n].val.clusterDim.y = 1;
    at[n].val.clusterDim.z = 1;
    ++n;
  }
  if (query_only) {
    cfg.attrs = at;
    cfg.numAttrs = n;
    if (g.ctas > num_sms) return RNN_ERR_LAUNCH;
    if (g.cluster > 1) {
      int nc = 0;
      if (cudaOccupancyMaxActiveClusters(&nc, k, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        return RNN_ERR_LAUNCH;
      }
      if (nc * g.cluster < g.ctas) return RNN_ERR_LAUNCH;
    } else {
      int per_sm = 0;
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, kThreads, dyn) != cudaSuccess) return RNN_ERR_CUDA;
      if (per_sm * num_sms < g.ctas) return RNN_ERR_LAUNCH;
    }
    return RNN_OK;
  }
  at[n].id = cudaLaunchAttributeCooperative;
  at[n].val.cooperative = 1;
  ++n;
  cfg.attrs = at;
  cfg.numAttrs = n;
  launch_begin(L);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, k, maps, a);
  launch_end(L);
  return cuda_status(e);
}

int dispatch(const Launch& L, int cell, const StackMaps& maps, const StackArgs& a, const Geom& g, bool query_only,
             int num_sms) {
#define RNN_S(C)                                                                          \
  if (cell == C) {                                                                        \
    if (g.N == 16) return launch_t<C, 16>(L, maps, a, g, query_only, num_sms);            \
    if (g.N == 32) return launch_t<C, 32>(L, maps, a, g, query_only, num_sms);            \
    return launch_t<C, 64>(L, maps, a, g, query_only, num_sms);                           \
  }
  RNN_S(LSTM) RNN_S(GRU) RNN_S(TANH) RNN_S(RELU)
#undef RNN_S
  return RNN_ERR_UNSUPPORTED;
}

}  // namespace

int stack_check(int cell, int H, int B, int nl, int first_p, int u_pack, int num_sms, int* ctas) {
  Geom g;
  RNN_TRY_LOCAL(geometry(cell, H, B, nl, first_p, &g));
  const int uc = cell == LSTM || cell == GRU ? 32 : 128;
  if (u_pack < 1 || uc % u_pack) return RNN_ERR_UNSUPPORTED;
  if (ctas) *ctas = g.ctas;
  if (num_sms <= 0) return g.ctas <= 152 ? RNN_OK : RNN_ERR_LAUNCH;  // host-side planning: GB300
  StackMaps maps{};
  StackArgs a{};
  Launch L{};
  return dispatch(L, cell, maps, a, g, true, num_sms);
}

int stack_fwd(const Launch& L, int cell, const StackArgs& in) {
  Geom g;
  const int rc = geometry(cell, in.H, in.B, in.nl, in.lay[0].P != nullptr, &g);
  if (rc != RNN_OK) return rc;
  StackArgs a = in;
  a.kc = g.kc;
  a.cluster = g.cluster;
  for (int l = 0; l < in.nl; ++l) {
    a.ks[l] = g.ks[l];
    a.kcx[l] = g.kcx[l];
    a.cta0[l] = g.cta0[l];
    a.ctas[l] = g.lctas[l];
  }
  a.cta0[in.nl] = g.cta0[in.nl];
  a.sm.a = g.sm.a;
  a.sm.ring = g.sm.ring;
  a.sm.rbuf = g.sm.rbuf;
  a.sm.smg = g.sm.smg;
  a.sm.smhn = g.sm.smhn;
  a.sm.bars = g.sm.bars;
  const int G = cell == LSTM ? 4 : cell == GRU ? 3 : 1;
  const int GH = G * in.H;
  StackMaps maps;
  memset(&maps, 0, sizeof(maps));
  for (int l = 0; l < in.nl; ++l) {
    const StackLayer& ly = in.lay[l];
    if (!ly.hseq || !ly.Wh) return RNN_ERR_INVALID_ARG;
    // weight rows: box of 64 k x 128 rows (rows past the end read zero)
    RNN_TRY_LOCAL(encode_operand(&maps.wh[l], Operand{ly.Wh, in.H, 0, GH, in.H}, 128));
    if (g.kcx[l]) {
      if (!ly.Wx || !ly.in || ly.In != in.H) return RNN_ERR_INVALID_ARG;
      RNN_TRY_LOCAL(encode_operand(&maps.wx[l], Operand{ly.Wx, in.H, 0, GH, in.H}, 128));
    } else if (!ly.P) {
      return RNN_ERR_INVALID_ARG;
    }
    // h sequence [T+1][B][H] as (T+1)*B rows: box of 64 k x N batch rows
    RNN_TRY_LOCAL(encode_operand(&maps.h[l + 1], Operand{ly.hseq, in.H, 0, (in.T + 1) * in.B, in.H}, g.N));
  }
  if (g.kcx[0]) RNN_TRY_LOCAL(encode_operand(&maps.h[0], Operand{in.lay[0].in, in.H, 0, (in.T + 1) * in.B, in.H}, g.N));
  return dispatch(L, cell, maps, a, g, false, L.num_sms);
}

}  // namespace rnn
