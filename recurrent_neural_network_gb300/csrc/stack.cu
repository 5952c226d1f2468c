// stack.cu -- persistent forward recurrence of a group of stacked layers for
// batches of up to 64 sequences, all timesteps in one launch.
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
//    [input | recurrent] in tensor memory for the whole launch (row i in
//    TMEM lane i, the A operand of every MMA): read from shared memory, the
//    128 KB block cost the tensor core ~270 ns per 64-deep K block whatever
//    the batch width, from TMEM it costs nothing extra.  The first layer of the
//    whole stack takes its input projection P = x W_x^T + b from one GEMM
//    over all timesteps and its K is the recurrent part only; every other
//    layer computes its input projection step by step from the layer
//    below's h_t (the K chunks of the input part), so a layer can start step
//    t as soon as the layer below has finished it.
//  * Per timestep a CTA waits for the arrival counter of what its chunk
//    reads (the layer below's step t for an input chunk, its own layer's
//    step t-1 for a recurrent chunk), then one thread streams the batch rows
//    of that chunk (N = batch rounded up to 16, x 64 k per block) from L2
//    into a ring of shared-memory stages with TMA (two timesteps deep where
//    it fits), and one thread issues tcgen05.mma (A from TMEM, M = 128 rows,
//    N, K = 16) into a double-buffered TMEM accumulator.
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
#include "stack.cuh"
#include "tc.cuh"

namespace rnn {

namespace {

using namespace stk;

// TMA maps of one launch over the h sequences, 3-D: (64 k of a block, batch
// row, k block) with box (64, N, kc / 64), so that one load brings a CTA's
// whole K chunk of a timestep (a TMA load costs ~150 ns to issue whatever
// its size, and 8 loads of 4-8 KB each per timestep were the bound).
struct StackMaps {
  CUtensorMap hx[kStackMaxLayers];  // layer l's input (the layer below's h sequence), box depth of layer l
  CUtensorMap hh[kStackMaxLayers];  // layer l's own h sequence, box depth of layer l
};

constexpr int kMaxStages = 4;  // input buffers, one timestep's K chunk each
constexpr int kThreads = 320;  // warp 0 TMA, warp 1 MMA, warps 2-9 epilogue (two per TMEM lane quadrant)

// Shared-memory layout of a CTA (offsets from the 1024-aligned base): the
// weights beyond what TMEM holds (kcs k of the 128 rows, 128-byte-swizzled
// K-major blocks of 128 x 64, the A operand of the MMAs that read it), the
// ring of input buffers (kc / 64 blocks of N x 64 bf16 each), the receive
// buffers of the cross-chunk reduction, the gate tile, barriers.
struct Smem {
  int a, ring, rbuf, smg, smhn, bars, total, stages;
};
__host__ __device__ inline Smem smem_layout(int cell, int N, int kc, int ksmin, int ksmax, int stages, int kcs = 0) {
  Smem s;
  s.a = 0;
  s.stages = stages;
  s.ring = 128 * kcs * 2;
  s.rbuf = s.ring + stages * (kc / 64) * N * 128;
  // [2][ksmax-1][N/ks/4][128] float4 for the largest ks of the launch (the
  // footprint (ks-1)/ks * N is largest for the largest ks)
  const int rb = ksmax > 1 ? 2 * (ksmax - 1) * (N / ksmax) * 128 * 4 : 0;
  s.smg = s.rbuf + rb;
  // gate tile [N/ks][128] and GRU recurrent candidate part [N/ks][32] for the
  // widest batch slice of the launch (smallest ks)
  s.smhn = s.smg + (N / ksmin) * 128 * 4;
  s.bars = s.smhn + (cell == GRU ? (N / ksmin) * 32 * 4 : 0);
  s.total = s.bars + 512;
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

// What the loops of one CTA read, copied once out of the launch arguments
// into registers: the arguments live in parameter space, and a field read
// there inside a loop that also stores to global memory is read again on
// every iteration (measured: ~150-270 ns per producer, MMA or epilogue
// iteration before this copy).
struct Run {
  int T, B, H, u_pack, kc, kct, cluster, test_skip_publish;
  int* err;
  uint64_t limit_ns;
  unsigned int* cnt;        // [layers][T] counters of the launch
  unsigned int want_h;      // CTAs of this CTA's layer
  unsigned int want_x;      // CTAs of the layer below (when it runs in this launch)
  StackSmem sm;
  StackLayer ly;            // this CTA's layer
};

__device__ __forceinline__ void abort_cluster(const Ctx& c, int cluster) { stk::abort_cluster(c.abort_flag, cluster); }
__device__ __forceinline__ bool wait_count(const unsigned int* cnt, unsigned int want, const Ctx& c, const Run& a) {
  return stk::wait_count(cnt, want, c.abort_flag, a.cluster, a.err, a.limit_ns);
}

// ---------------------------------------------------------------------------
// epilogue: 256 threads, two halves of four warps (one warp per TMEM lane
// quadrant in each).  Thread (row, hf) owns packed row `row` of the CTA's
// block for the columns [hf*NH, hf*NH + NH) of this CTA's batch slice
// [me*NS, me*NS + NS) (NH = NS/2; with NS < 8 the first half takes all NS);
// in the cell update thread e takes unit j0 + lane and slice columns
// 8 i + e / 32.  Two warps per scheduler halve every loop of the epilogue
// and leave a second warp to issue while one waits.
template <int CELL, int N, int KS>
__device__ void epilogue(const Run& a, const Ctx& c, int row, int hf, int e, uint32_t acc_base) {
  constexpr int G = CellInfo<CELL>::G;
  constexpr bool SIMPLE = G == 1;
  constexpr int UC = SIMPLE ? 128 : 32;
  constexpr int ROWS = G * UC;
  constexpr int NS = N / KS;
  constexpr bool TWO = NS >= 8;               // both halves take columns
  constexpr int NH = TWO ? NS / 2 : NS;       // columns of a half
  constexpr int PP = SIMPLE ? 1 : (NS + 7) / 8;  // (unit, batch column) pairs per thread
  constexpr int NC4 = NS / 4;                 // float4 chunks of a slice
  constexpr bool SPLIT = CELL == GRU;         // input and recurrent sums apart (GRU candidate gate)
  constexpr int ACC = N < 32 ? 32 : N;        // TMEM columns between the two accumulators
  const StackLayer& ly = a.ly;
  const int T = a.T, B = a.B, H = a.H, GH = G * H, u = a.u_pack;
  const int me = c.me, kcx = c.kcx;
  const int j0 = c.rb * UC, r0 = j0 * G;
  const int lane = threadIdx.x & 31, w8 = e >> 5;
  const bool act = TWO || hf == 0;            // this half takes columns
  const int c0h = hf * NH;                    // first slice column of this half
  const int cb = me * NS + c0h;               // its first batch entry
  const uint32_t lane_q = static_cast<uint32_t>(row & ~31) << 16;
  const bool live_row = row < ROWS;
  // gate and unit of this thread's row
  const int rg = (row % (G * u)) / u;
  const int rj = (row / (G * u)) * u + row % u;
  const float bias = (live_row && !ly.P) ? ly.bias[r0 + row] : 0.f;
  const float bias_hn = (CELL == GRU && live_row && rg == 2) ? ly.bias_hn[j0 + rj] : 0.f;
  // gate activation of this row as ga * tanh(ga * x) + gc: sigmoid (input,
  // forget, output, reset, update) or tanh (LSTM cell candidate)
  const bool is_tanh = CELL == LSTM && rg == 2;
  const float ga = is_tanh ? 1.f : 0.5f, gc = is_tanh ? 0.f : 0.5f;
  float* const gout = ly.gates_out;
  // rows of the G gates of unit j0 + lane in the gate tile (cell update)
  const int o0 = packed_row(0, lane, G, u), o1 = packed_row(G > 1 ? 1 : 0, lane, G, u);
  const int o2 = packed_row(G > 2 ? 2 : 0, lane, G, u), o3 = packed_row(G > 3 ? 3 : 0, lane, G, u);
  float* smg = reinterpret_cast<float*>(c.smem + a.sm.smg);
  float* smhn = reinterpret_cast<float*>(c.smem + a.sm.smhn);
  float4* rbuf = reinterpret_cast<float4*>(c.smem + a.sm.rbuf);
  // receive buffer of parity p from the peer in slot s: [p][s][chunk][row]
  auto rb_at = [&](int p, int s, int ch) -> float4* { return rbuf + ((p * (KS - 1) + s) * NC4 + ch) * 128; };

  // per-pair state (LSTM c, GRU h_{t-1}) kept across steps
  float st[PP];
#pragma unroll
  for (int i = 0; i < PP; ++i) {
    st[i] = 0.f;
    if constexpr (!SIMPLE) {
      const int cc = 8 * i + w8, b = me * NS + cc;
      if (cc < NS && b < B) {
        if (CELL == LSTM && ly.c0) st[i] = ly.c0[(size_t)b * H + j0 + lane];
        if (CELL == GRU) st[i] = __bfloat162float(ly.hseq[(size_t)b * H + j0 + lane]);
      }
    }
  }

  for (int t = 0; t < T; ++t) {
    const int acc = t & 1, par = t & 1;
    const uint32_t ph = (uint32_t)(t >> 1) & 1u;
    if (KS > 1 && e == 0) tc::mbar_arrive_expect_tx(&c.rbar[par], (uint32_t)((KS - 1) * 128 * NS * 4));
    // sx: input part (the first layer's input projection P, loaded before the
    // accumulator is ready, or the folded bias plus the input chunks); sh:
    // recurrent part (GRU only: the other cells add everything into sx).  P
    // is loaded unconditionally from clamped addresses (a loaded value
    // selected against 0 is consumed at the select, which made each column's
    // load wait for the previous one); columns past the batch and rows past
    // the block are never stored.
    float sx[NH], sh[SPLIT ? NH : 1];
    if (ly.P) {
      const float* prow = ly.P + (size_t)t * B * GH + min(r0 + row, GH - 1);
#pragma unroll
      for (int cc = 0; cc < NH; ++cc) sx[cc] = prow[(size_t)min(cb + cc, B - 1) * GH];
    } else {
#pragma unroll
      for (int cc = 0; cc < NH; ++cc) sx[cc] = bias;
    }
#pragma unroll
    for (int cc = 0; cc < (SPLIT ? NH : 0); ++cc) sh[cc] = 0.f;
    // ---- accumulator of this step: this half's columns of every chunk's
    // slice, its own added to the sums, the others sent to their owners
    bool ok;
    {
      int w = 1;
      if (lane == 0) w = tc::mbar_wait(&c.tfull[acc], ph, c.abort_flag, a.err, a.limit_ns) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, w, 0) != 0;
    }
    if (ok) {
      tc::fence_after_sync();
      if (act) {
        constexpr int NL = NH < 16 ? NH : 16;  // columns per TMEM load
#pragma unroll
        for (int p = 0; p < KS; ++p) {
#pragma unroll
          for (int l0 = 0; l0 < NH; l0 += NL) {
            float w[NL];
            tc::tmem_load_cols<NL>(c.tmem + lane_q + acc_base + (uint32_t)(acc * ACC + p * NS + c0h + l0), w);
            if (p == me) {
#pragma unroll
              for (int q = 0; q < NL; ++q) {
                if (SPLIT && me >= kcx) sh[SPLIT ? l0 + q : 0] += w[q];
                else sx[l0 + q] += w[q];
              }
            } else if constexpr (KS > 1) {
              const int slot = me < p ? me : me - 1;
              const uint32_t prank = (uint32_t)(c.crank - me + p);
              const uint32_t bar = tc::mapa(tc::smem_addr(&c.rbar[par]), prank);
#pragma unroll
              for (int q = 0; q < NL / 4; ++q)
                st_async_v4(tc::mapa(tc::smem_addr(rb_at(par, slot, (c0h + l0) / 4 + q) + row), prank), w + 4 * q,
                            bar);
            }
          }
        }
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&c.tempty[acc]);
      if constexpr (KS > 1) {
        int w = 1;
        if (lane == 0) w = wait_cluster_bytes(&c.rbar[par], ph, c.abort_flag, a.err, a.limit_ns) ? 1 : 0;
        ok = __shfl_sync(0xffffffffu, w, 0) != 0;
      }
    }
    if (!ok && lane == 0) {
      *c.ep_fail = 1;
      abort_cluster(c, a.cluster);
    }
    tc::named_bar(1, 256);
    if (*reinterpret_cast<volatile int*>(c.ep_fail)) break;

    // ---- the other chunks' partial sums of this half's columns, in chunk
    // order (input and recurrent parts apart for GRU)
    if (act) {
#pragma unroll
      for (int k = 0; k < KS; ++k) {
        if (k == me) continue;
        const bool xk = !SPLIT || k < kcx;
        const int slot = k < me ? k : k - 1;
#pragma unroll
        for (int q = 0; q < NH / 4; ++q) {
          const float4 v = rb_at(par, slot, c0h / 4 + q)[row];
          const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            if (SPLIT && !xk) sh[SPLIT ? 4 * q + i : 0] += vv[i];
            else sx[4 * q + i] += vv[i];
          }
        }
      }
    }

    // ---- gates of this row for this half's columns (branch-free: sigmoid
    // is ga * tanh(ga x) + gc; column bounds only guard the global stores)
    const size_t tb = (size_t)t * B;
    const int nval = (live_row && act) ? min(NH, B - cb) : 0;
    if constexpr (!SIMPLE) {
      if (act) {
        float gv[NH];
#pragma unroll
        for (int cc = 0; cc < NH; ++cc) {
          const float x = SPLIT ? sx[cc] + sh[SPLIT ? cc : 0] : sx[cc];
          gv[cc] = fmaf(ga, tanh_hw(ga * x), gc);
          if constexpr (SPLIT) gv[cc] = rg == 2 ? sx[cc] : gv[cc];  // GRU candidate row: x_n + b_xn
        }
#pragma unroll
        for (int cc = 0; cc < NH; ++cc) smg[(c0h + cc) * 128 + row] = gv[cc];
        if constexpr (SPLIT) {
          if (live_row && rg == 2) {
#pragma unroll
            for (int cc = 0; cc < NH; ++cc) smhn[(c0h + cc) * 32 + rj] = sh[SPLIT ? cc : 0] + bias_hn;
          }
        }
        if (gout && (!SPLIT || rg < 2)) {
          float* const go = gout + (tb + cb) * GH + r0 + row;
#pragma unroll
          for (int cc = 0; cc < NH; ++cc)
            if (cc < nval) go[(size_t)cc * GH] = gv[cc];
        }
      }
    } else {
      // simple RNN: the row is the unit, h = act(x) directly
      if (act) {
        float hv[NH];
#pragma unroll
        for (int cc = 0; cc < NH; ++cc) hv[cc] = simple_act<CELL, __nv_bfloat16>(sx[cc]);
        __nv_bfloat16* const hs = ly.hseq + ((size_t)(t + 1) * B + cb) * H + j0 + row;
        __nv_bfloat16* const ys = ly.y ? ly.y + (tb + cb) * H + j0 + row : nullptr;
        __nv_bfloat16* const hTs = (t == T - 1 && ly.hT) ? ly.hT + (size_t)cb * H + j0 + row : nullptr;
        float* const go = gout ? gout + (tb + cb) * GH + r0 + row : nullptr;
#pragma unroll
        for (int cc = 0; cc < NH; ++cc) {
          if (cc >= nval) break;
          const __nv_bfloat16 hb = __float2bfloat16_rn(hv[cc]);
          hs[(size_t)cc * H] = hb;
          if (ys) ys[(size_t)cc * H] = hb;
          if (hTs) hTs[(size_t)cc * H] = hb;
          if (go) go[(size_t)cc * GH] = hv[cc];
        }
      }
    }
    if constexpr (!SIMPLE) {
      tc::named_bar(1, 256);
      // ---- cell update of this thread's (unit, batch column) pairs: unit
      // j0 + lane, slice column cc = 8 i + w8; arithmetic first, then the
      // stores, so that the pairs' latencies overlap
      float hv[PP], nv[SPLIT ? PP : 1], hnv[SPLIT ? PP : 1];
#pragma unroll
      for (int i = 0; i < PP; ++i) {
        const int cc = min(8 * i + w8, NS - 1);  // pairs past the slice compute on column NS-1 and store nothing
        const float* gr = smg + cc * 128;
        if constexpr (CELL == LSTM) {
          float ig, fg, gg, og;
          if (u == 1) {
            const float4 g4 = *reinterpret_cast<const float4*>(gr + 4 * lane);
            ig = g4.x; fg = g4.y; gg = g4.z; og = g4.w;
          } else {
            ig = gr[o0]; fg = gr[o1]; gg = gr[o2]; og = gr[o3];
          }
          st[i] = fmaf(fg, st[i], ig * gg);
          hv[i] = og * tanh_hw(st[i]);
        } else {
          const float r = gr[o0], z = gr[o1], xn = gr[o2];
          const float hn = smhn[cc * 32 + lane];
          const float n = tanh_hw(fmaf(r, hn, xn));
          hv[i] = fmaf(z, st[i] - n, n);  // (1 - z) n + z h_{t-1}
          st[i] = hv[i];
          nv[SPLIT ? i : 0] = n;
          hnv[SPLIT ? i : 0] = hn;
        }
      }
      // stores: slice column cc is batch entry me * NS + cc
      const int bb = me * NS + w8;  // batch entry of pair 0
      auto okp = [&](int i) { return 8 * i + w8 < NS && bb + 8 * i < B; };
      const size_t off = (size_t)bb * H + j0 + lane;
      __nv_bfloat16* const hs = ly.hseq + (size_t)(t + 1) * B * H + off;
#pragma unroll
      for (int i = 0; i < PP; ++i)
        if (okp(i)) hs[(size_t)(8 * i) * H] = __float2bfloat16_rn(hv[i]);
      if (ly.y) {
        __nv_bfloat16* const ys = ly.y + tb * H + off;
#pragma unroll
        for (int i = 0; i < PP; ++i)
          if (okp(i)) ys[(size_t)(8 * i) * H] = __float2bfloat16_rn(hv[i]);
      }
      if (t == T - 1 && ly.hT) {
#pragma unroll
        for (int i = 0; i < PP; ++i)
          if (okp(i)) ly.hT[off + (size_t)(8 * i) * H] = __float2bfloat16_rn(hv[i]);
      }
      if constexpr (CELL == LSTM) {
        if (ly.c_out) {
          float* const cs = ly.c_out + tb * H + off;
#pragma unroll
          for (int i = 0; i < PP; ++i)
            if (okp(i)) cs[(size_t)(8 * i) * H] = st[i];
        }
        if (t == T - 1 && ly.cT) {
#pragma unroll
          for (int i = 0; i < PP; ++i)
            if (okp(i)) ly.cT[off + (size_t)(8 * i) * H] = st[i];
        }
      } else {
        if (gout) {
          float* const gs = gout + (tb + bb) * GH + r0 + o2;
#pragma unroll
          for (int i = 0; i < PP; ++i)
            if (okp(i)) gs[(size_t)(8 * i) * GH] = nv[SPLIT ? i : 0];
        }
        if (ly.hn_out) {
          float* const hns = ly.hn_out + tb * H + off;
#pragma unroll
          for (int i = 0; i < PP; ++i)
            if (okp(i)) hns[(size_t)(8 * i) * H] = hnv[SPLIT ? i : 0];
        }
      }
    }
    // ---- publish h_t of this CTA's units and batch slice: the readers load
    // it with TMA (async proxy) after acquiring the counter
    tc::fence_proxy_async_global();
    tc::named_bar(1, 256);
    if (e == 0 && !(a.test_skip_publish && blockIdx.x == 0 && t == 0))
      red_release_add_u32(a.cnt + (size_t)c.li * T + t, 1u);
  }
}

template <int CELL, int N>
__global__ void __launch_bounds__(kThreads, 1)
    stack_fwd_kernel(const __grid_constant__ StackMaps maps, const __grid_constant__ StackArgs p) {
  constexpr int G = CellInfo<CELL>::G;
  constexpr int UC = G == 1 ? 128 : 32;
  constexpr int RING = N * 128;
  constexpr uint32_t TMEM_COLS = 512;  // weights (kct / 2 columns) + two accumulators
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (p.cluster > 1) {
    uint32_t ncta;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(ncta));
    if ((int)ncta != p.cluster) {
      if (threadIdx.x == 0) raise_error(p.err, DEV_BAD_CLUSTER);
      return;
    }
  }
  int li = 0;
  while (li + 1 < p.nl && (int)blockIdx.x >= p.cta0[li + 1]) ++li;
  Run a;
  a.T = p.T;
  a.B = p.B;
  a.H = p.H;
  a.u_pack = p.u_pack;
  a.kc = p.kcl[li];
  a.kct = p.kctl[li];
  a.cluster = p.cluster;
  a.test_skip_publish = p.test_skip_publish;
  a.err = p.err;
  a.limit_ns = p.limit_ns;
  a.cnt = p.cnt;
  a.want_h = (unsigned)p.ctas[li];
  a.want_x = li > 0 ? (unsigned)p.ctas[li - 1] : 0u;
  a.sm = p.sm;
  a.ly = p.lay[li];
  const int NST = a.sm.stages;
  Ctx c;
  c.smem = smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + a.sm.bars);
  c.full = bars;
  c.empty = c.full + kMaxStages;
  c.tfull = c.empty + kMaxStages;
  c.tempty = c.tfull + 2;
  c.rbar = c.tempty + 2;
  c.abar = c.rbar + 2;
  c.dbar = c.abar + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(c.dbar + 1);
  c.abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  c.ep_fail = reinterpret_cast<int*>(tmem_slot + 2);
  c.li = li;
  c.ks = p.ks[li];
  c.kcx = p.kcx[li];
  const int local = (int)blockIdx.x - p.cta0[li];
  c.rb = local / c.ks;
  c.me = local % c.ks;
  c.crank = a.cluster > 1 ? (int)tc::cluster_ctarank() : 0;
  const StackLayer& ly = a.ly;
  const bool xpart = c.me < c.kcx;
  const int k0 = (xpart ? c.me : c.me - c.kcx) * a.kc;
  const int nkb = a.kc / 64;
  const int r0 = c.rb * UC * G;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NST; ++s) {
      tc::mbar_init(c.full + s, 1);
      tc::mbar_init(c.empty + s, 1);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(c.tfull + i, 1);
      tc::mbar_init(c.tempty + i, 8);
      tc::mbar_init(c.rbar + i, 1);
    }
    tc::mbar_init(c.abar, 8);  // the eight epilogue warps, once their share of the weights is in TMEM
    tc::mbar_init(c.dbar, 1);
    *c.abort_flag = 0;
    *c.ep_fail = 0;
    tc::fence_mbar_init();
    tc::tma_prefetch_desc(xpart ? &maps.hx[c.li] : &maps.hh[c.li]);
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
  // TMEM columns: [0, kct/2) this CTA's block of weight rows (row i in lane
  // i, two consecutive k per column), then the two accumulators; k from kct
  // to kc (if any) in shared memory
  const uint32_t acc_base = (uint32_t)(a.kct / 2);

  int last_par[kMaxStages];  // producer: parity of the last load issued into each buffer (-1: none)
  for (int s = 0; s < kMaxStages; ++s) last_par[s] = -1;
  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      const CUtensorMap* src = xpart ? &maps.hx[c.li] : &maps.hh[c.li];
      for (int t = 0; t < a.T; ++t) {
        bool ok = true;
        if (xpart) {
          if (ly.wait_in) ok = wait_count(a.cnt + (size_t)(c.li - 1) * a.T + t, a.want_x, c, a);
        } else if (t > 0) {
          ok = wait_count(a.cnt + (size_t)c.li * a.T + t - 1, a.want_h, c, a);
        }
        if (!ok) break;
        // h written by other CTAs' generic stores, read here through the async proxy
        tc::fence_proxy_async_global();
        const int slot = xpart ? t + 1 : t;
        // the whole K chunk of this timestep in one load: nkb blocks of N
        // batch rows x 64 k, laid out one block after the other
        if (!tc::mbar_wait(c.empty + stage, phase ^ 1, c.abort_flag, a.err, a.limit_ns)) break;
        tc::mbar_arrive_expect_tx(c.full + stage, (uint32_t)(nkb * RING));
        last_par[stage] = (int)phase;
        tc::tma_load_3d(smem + a.sm.ring + stage * nkb * RING, src, c.full + stage, 0, slot * a.B, k0 / 64);
        if (++stage == (uint32_t)NST) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (*c.abort_flag) abort_cluster(c, a.cluster);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = tc::idesc_bf16(128, N, 0, 0);
      const int nkt = a.kct / 64;
      const uint64_t ad0 = tc::sdesc_sw128(tc::smem_addr(smem + a.sm.a), 16, 1024);
      bool ok = tc::mbar_wait(c.abar, 0, c.abort_flag, a.err, a.limit_ns);
      tc::fence_after_sync();
      uint32_t stage = 0, phase = 0;
      for (int t = 0; t < a.T && ok; ++t) {
        const int acc = t & 1;
        if (!tc::mbar_wait(c.tempty + acc, ((uint32_t)(t >> 1) & 1u) ^ 1u, c.abort_flag, a.err, a.limit_ns)) break;
        tc::fence_after_sync();
        const uint32_t d = c.tmem + acc_base + (uint32_t)(acc * (N < 32 ? 32 : N));
        if (!tc::mbar_wait(c.full + stage, phase, c.abort_flag, a.err, a.limit_ns)) break;
        tc::fence_after_sync();
        const uint32_t sb0 = tc::smem_addr(smem + a.sm.ring + stage * nkb * RING);
        // descriptors stepped in their 16-byte address field (one 64-k block
        // of the buffer is RING bytes, one 16-k step 32 bytes; the field
        // does not carry out for shared-memory addresses), the first MMA
        // overwriting the accumulator
        const uint64_t bd0 = tc::sdesc_sw128(sb0, 16, 1024);
        tc::mma_bf16_ta(d, c.tmem, bd0, idesc, 0u);
#pragma unroll
        for (int i = 1; i < 4 * 14; ++i) {
          if (i >= 4 * nkt) break;
          const int kb = i >> 2, kk = i & 3;
          tc::mma_bf16_ta(d, c.tmem + (uint32_t)(8 * i), bd0 + (uint64_t)((kb * RING + kk * 32) >> 4), idesc, 1u);
        }
        // the k blocks past kct: A from the swizzled blocks in shared memory
        for (int i = 0; i < 4 * (nkb - nkt); ++i) {
          const int kb = nkt + (i >> 2), kk = i & 3;
          tc::mma_bf16(d, ad0 + (uint64_t)(((i >> 2) * 16384 + kk * 32) >> 4),
                       bd0 + (uint64_t)((kb * RING + kk * 32) >> 4), idesc, 1u);
        }
        tc::mma_commit(c.empty + stage);
        if (++stage == (uint32_t)NST) {
          stage = 0;
          phase ^= 1;
        }
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
    const int hf = (warp - 2) >> 2;  // half of the epilogue (two warps per TMEM lane quadrant)
    const int e = threadIdx.x - 64;
    {
      // this row of the CTA's weight block into TMEM, the two halves taking
      // alternate 32-wide k blocks (rows past the block's gate rows, GRU's
      // last 32, hold zeros)
      const int G_H = G * a.H;
      const bool live = row < G * UC && r0 + row < G_H;
      const __nv_bfloat16* wrow = (xpart ? ly.Wx : ly.Wh) + (size_t)(r0 + row) * a.H + k0;
      const uint32_t lane_q = static_cast<uint32_t>(row & ~31) << 16;
      for (int c16 = hf; c16 < a.kct / 32; c16 += 2) {
        float v[16];
        if (live) {
          const uint4* q = reinterpret_cast<const uint4*>(wrow + c16 * 32);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint4 u = q[i];
            v[4 * i] = __uint_as_float(u.x);
            v[4 * i + 1] = __uint_as_float(u.y);
            v[4 * i + 2] = __uint_as_float(u.z);
            v[4 * i + 3] = __uint_as_float(u.w);
          }
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) v[i] = 0.f;
        }
        tc::tmem_store16(c.tmem + lane_q + (uint32_t)(c16 * 16), v);
      }
      // k past kct into shared memory as K-major 128 x 64 blocks with the
      // 128-byte swizzle (16-byte piece q of row r at piece q ^ (r % 8)),
      // the layout a TMA load with that swizzle would write
      for (int q8 = hf; q8 < (a.kc - a.kct) / 8; q8 += 2) {
        const uint4 u = live ? *reinterpret_cast<const uint4*>(wrow + a.kct + q8 * 8) : make_uint4(0, 0, 0, 0);
        const int blk = q8 >> 3, q = q8 & 7;
        *reinterpret_cast<uint4*>(smem + a.sm.a + blk * 16384 + row * 128 + ((q ^ (row & 7)) << 4)) = u;
      }
      tc::fence_proxy_async_smem();  // generic stores read by the tensor core (async proxy)
      tc::tmem_store_wait();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(c.abar);
    }
    if (c.ks == 1) epilogue<CELL, N, 1>(a, c, row, hf, e, acc_base);
    else if (c.ks == 2) epilogue<CELL, N, 2>(a, c, row, hf, e, acc_base);
    else epilogue<CELL, N, 4>(a, c, row, hf, e, acc_base);
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0 && lane == 0 && *c.abort_flag) {
    // copies already issued land before the CTA's shared memory goes away
    // (after an abort some were never consumed)
    for (int s = 0; s < NST; ++s) {
      if (last_par[s] < 0) continue;
      const uint64_t t0 = globaltimer_ns();
      while (!tc::mbar_try_wait(c.full + s, (uint32_t)last_par[s]) && globaltimer_ns() - t0 < 1000000ull) {
      }
    }
  }
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(c.tmem, TMEM_COLS);
  }
  if (a.cluster > 1) tc::cluster_sync_all();  // no peer stores into this CTA's shared memory after it exits
}

// Geometry of a launch over layers [0, nl) of a group: K chunk width and
// chunks per layer, CTAs.  first_p: the group's first layer reads P (it is
// the stack's layer 0, K = H; the others have K = 2H).  A CTA's epilogue
// works on N / ks batch columns, and the wavefront moves at the pace of its
// slowest layer, so chunks are narrowed (512 -> 256) on the layers with the
// fewest chunks while the CTAs stay within `budget`.  Where the group does
// not fit the budget with 512-wide chunks, the layers with the most chunks
// are widened to 1024 (H a multiple of 1024): such a chunk keeps what fits
// beside the accumulators in TMEM (kct) and the rest in shared memory.
struct Geom {
  int N, cluster, ctas;
  int kc[kStackMaxLayers], kct[kStackMaxLayers], ks[kStackMaxLayers], kcx[kStackMaxLayers],
      cta0[kStackMaxLayers + 1], lctas[kStackMaxLayers];
  Smem sm;
};

int geometry(int cell, int H, int B, int nl, int first_p, int budget, Geom* g) {
  if (nl < 1 || nl > kStackMaxLayers || B < 1 || B > 64) return RNN_ERR_UNSUPPORTED;
  const int G = cell == LSTM ? 4 : cell == GRU ? 3 : 1;
  const int uc = G == 1 ? 128 : 32;
  if (H % uc || H % 256) return RNN_ERR_UNSUPPORTED;
  g->N = B <= 16 ? 16 : B <= 32 ? 32 : 64;
  const int rbs = H / uc;
  // TMEM columns beside two accumulators of N (at least 32) columns: two k per column
  const int kt_max = 2 * (512 - 2 * (g->N < 32 ? 32 : g->N));
  auto set = [&](int l, int kc) {
    const bool p = l == 0 && first_p;
    g->kc[l] = kc;
    g->kct[l] = std::min(kc, kt_max / 64 * 64);
    g->kcx[l] = p ? 0 : H / kc;  // layers above the first: input width H
    g->ks[l] = g->kcx[l] + H / kc;
  };
  int cta = 0;
  for (int l = 0; l < nl; ++l) {
    set(l, H % 512 == 0 ? 512 : 256);
    if (g->ks[l] != 1 && g->ks[l] != 2 && g->ks[l] != 4) return RNN_ERR_UNSUPPORTED;
    if (g->N / g->ks[l] < 4) return RNN_ERR_UNSUPPORTED;
    cta += rbs * g->ks[l];
  }
  // widen the layers with the most chunks while the group exceeds the budget
  while (cta > budget && H % 1024 == 0) {
    int kmax = 0, lw = -1;
    for (int l = 0; l < nl; ++l)
      if (g->kc[l] == 512 && g->ks[l] > kmax) kmax = g->ks[l], lw = l;
    if (lw < 0) break;
    cta -= rbs * g->ks[lw];
    set(lw, 1024);
    cta += rbs * g->ks[lw];
  }
  if (cta > budget) return RNN_ERR_LAUNCH;
  // narrow the chunks of every layer that has the fewest, while they fit
  for (;;) {
    int kmin = 8;
    for (int l = 0; l < nl; ++l) kmin = std::min(kmin, g->ks[l]);
    int extra = 0;
    bool can = true;
    for (int l = 0; l < nl; ++l) {
      if (g->ks[l] != kmin) continue;
      if (g->kc[l] != 512 || 2 * g->ks[l] > 4 || g->N / (2 * g->ks[l]) < 8) can = false;
      extra += rbs * g->ks[l];
    }
    if (!can || cta + extra > budget) break;
    for (int l = 0; l < nl; ++l)
      if (g->ks[l] == kmin) set(l, 256);
    cta += extra;
  }
  int ksmax = 1, ksmin = 4, kcmax = 0, kcsmax = 0;
  cta = 0;
  for (int l = 0; l < nl; ++l) {
    ksmax = std::max(ksmax, g->ks[l]);
    ksmin = std::min(ksmin, g->ks[l]);
    kcmax = std::max(kcmax, g->kc[l]);
    kcsmax = std::max(kcsmax, g->kc[l] - g->kct[l]);
    g->cta0[l] = cta;
    g->lctas[l] = rbs * g->ks[l];
    cta += g->lctas[l];
  }
  g->cta0[nl] = cta;
  g->ctas = cta;
  g->cluster = ksmax;
  for (int l = 0; l < nl; ++l)
    if (g->lctas[l] % ksmax) return RNN_ERR_UNSUPPORTED;
  // input buffers: two where they fit (a chunk whose input is ready early
  // loads the next step while this one computes)
  bool fit = false;
  for (int st : {2, 1}) {
    g->sm = smem_layout(cell, g->N, kcmax, ksmin, ksmax, st, kcsmax);
    if (g->sm.total + 1024 <= 227 * 1024) {
      fit = true;
      break;
    }
  }
  if (!fit) return RNN_ERR_UNSUPPORTED;
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

int stack_check(int cell, int H, int B, int nl, int first_p, int u_pack, int num_sms, int* ctas, int* wide) {
  Geom g;
  if (wide) *wide = 0;
  RNN_TRY_LOCAL(geometry(cell, H, B, nl, first_p, num_sms > 0 ? num_sms : 152, &g));
  if (wide)
    for (int l = 0; l < nl; ++l) *wide |= g.kc[l] > g.kct[l] ? 1 : 0;
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
  const int rc = geometry(cell, in.H, in.B, in.nl, in.lay[0].P != nullptr, L.num_sms > 0 ? L.num_sms : 152, &g);
  if (rc != RNN_OK) return rc;
  StackArgs a = in;
  a.cluster = g.cluster;
  for (int l = 0; l < in.nl; ++l) {
    a.kcl[l] = g.kc[l];
    a.kctl[l] = g.kct[l];
    a.ks[l] = g.ks[l];
    a.kcx[l] = g.kcx[l];
    a.cta0[l] = g.cta0[l];
    a.ctas[l] = g.lctas[l];
  }
  a.cta0[in.nl] = g.cta0[in.nl];
  a.sm.stages = g.sm.stages;
  a.sm.a = g.sm.a;
  a.sm.ring = g.sm.ring;
  a.sm.rbuf = g.sm.rbuf;
  a.sm.smg = g.sm.smg;
  a.sm.smhn = g.sm.smhn;
  a.sm.bars = g.sm.bars;
  StackMaps maps;
  memset(&maps, 0, sizeof(maps));
  for (int l = 0; l < in.nl; ++l) {
    const StackLayer& ly = in.lay[l];
    if (!ly.hseq || !ly.Wh) return RNN_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(ly.Wh) & 15) return RNN_ERR_INVALID_ARG;
    if (g.kcx[l]) {
      if (!ly.Wx || !ly.in || ly.In != in.H || (reinterpret_cast<uintptr_t>(ly.Wx) & 15)) return RNN_ERR_INVALID_ARG;
    } else if (!ly.P) {
      return RNN_ERR_INVALID_ARG;
    }
    // h sequences [T+1][B][H] as (T+1)*B rows, boxes of this layer's chunk depth
    const long long rows = (long long)(in.T + 1) * in.B;
    RNN_TRY_LOCAL(encode_seq3(&maps.hh[l], ly.hseq, rows, in.H, g.N, g.kc[l] / 64));
    if (g.kcx[l]) {
      const __nv_bfloat16* src = l == 0 ? ly.in : in.lay[l - 1].hseq;
      RNN_TRY_LOCAL(encode_seq3(&maps.hx[l], src, rows, in.H, g.N, g.kc[l] / 64));
    }
  }
  return dispatch(L, cell, maps, a, g, false, L.num_sms);
}

}  // namespace rnn
