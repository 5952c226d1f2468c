// stack_bwd.cu -- persistent backward-through-time of a group of stacked
// layers for batches of up to 64 sequences, all reverse timesteps of
// every layer of the group in one launch.
//
// "Persistent RNNs: Stashing Recurrent Weights On-Chip" (citing snippets on
// its page): the recurrent weights stay on chip across timesteps and one
// launch runs the whole sequence.  "Optimizing Performance of RNNs on GPUs"
// (review page, proposed method): the backward passes of consecutive layers
// overlap, layer l working on reverse step s while layer l+1 works on s-1.
//
// The gradient reaching h^l_s is dh^l_s = dGh^l_{s+1} W_h^l (own recurrence)
// + dGx^{l+1}_s W_x^{l+1} (the layer above; the user's dy at the top of the
// stack), a product of the gate gradients with the transposed weights:
//
//  * A CTA owns 128 hidden units (its 128 TMEM lanes) and one K chunk of the
//    layer's K = [G*H recurrent | G*H from above]: the transposed columns of
//    W_h^l or W_x^{l+1} for its units, resident in tensor memory for the
//    launch.  Per reverse step it waits for the arrival counter of what its
//    chunk reads (its own layer's step s+1, or the layer above's step s),
//    loads the batch rows of that chunk of dGh^l_{s+1} or dGx^{l+1}_s with
//    one 3-D TMA load, and one thread issues the tcgen05.mma products into a
//    double-buffered TMEM accumulator.  At s = T-1 the recurrent rows lie
//    past the end of dGh (read as zero by TMA), and so do the above rows at
//    the extra step s = -1, which computes dh0 = dGh^l_0 W_h^l.
//  * The K chunks of a unit block form a cluster and reduce-scatter their
//    partial sums over the batch (asynchronous stores into each other's
//    shared memory, summed in chunk order), so each CTA ends with dh for its
//    128 units and its slice of the batch: one (unit, batch column) per
//    thread and column, the layout the pointwise step needs.  That step (the
//    cell's derivative; its inputs -- gates, c, the GRU candidate's
//    recurrent part, h_{s-1}, dy -- are loaded before the accumulator is
//    ready) writes dGx (and, for GRU, dGh) in bf16, keeps the carried state
//    (LSTM dc, GRU dh z) in registers, and one release arrival per CTA
//    publishes step s of its layer.
//
// Every wait is bounded; a CTA that gives up records the error, aborts its
// cluster and leaves, as in the forward kernel (stack.cu).
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

// TMA maps per layer: the recurrent source dGh^l and the source from above
// dGx^{l+1}, each [T*B rows][G*H] with box (64, N, kc / 64).
struct BwdMaps {
  CUtensorMap rec[kStackMaxLayers];
  CUtensorMap above[kStackMaxLayers];
};

constexpr int kBufs = 2;        // input buffers, one timestep's K chunk each
constexpr int kThreads = 320;   // warp 0 TMA, warp 1 MMA, warps 2-9 epilogue (two per TMEM lane quadrant)
constexpr int kUnits = 128;     // hidden units per CTA (TMEM lanes)

// shared memory: the weights past what TMEM holds (kcs k of the 128 rows,
// 128-byte-swizzled K-major 128 x 64 blocks), input buffers, receive buffers
// of the reduction, barriers
struct BSmem {
  int a, ring, rbuf, bars, total, bufs;
};
inline BSmem bwd_layout(int N, int kcmax, int ksmax, int bufs, int kcs = 0) {
  BSmem s;
  s.bufs = bufs;
  s.a = 0;
  s.ring = 128 * kcs * 2;
  s.rbuf = s.ring + bufs * (kcmax / 64) * N * 128;
  const int rb = ksmax > 1 ? 2 * (ksmax - 1) * (N / ksmax) * 128 * 4 : 0;
  s.bars = s.rbuf + rb;
  s.total = s.bars + 512;
  return s;
}

struct BCtx {
  uint8_t* smem;
  uint64_t *full, *empty, *tfull, *tempty, *rbar, *abar, *dbar;
  uint32_t tmem;
  volatile int* abort_flag;
  int* ep_fail;
  int li, ub, me, ks, kr, crank;
};

// loop-invariant arguments of one CTA, in registers (see stack.cu: a field
// of the launch arguments read inside a loop is read again every iteration)
struct BRun {
  int T, B, H, u_pack, kc, kct, cluster, test_skip_publish;
  int* err;
  uint64_t limit_ns;
  unsigned int* cnt;
  unsigned int want_own, want_above;
  StackSmem sm;
  StackBwdLayer ly;
};

// ---------------------------------------------------------------------------
// epilogue: 256 threads in two halves of four warps; thread (row, hf) owns
// hidden unit j = 128 ub + row (TMEM lane row) for the columns [hf*NH,
// hf*NH + NH) of this CTA's batch slice [me*NS, me*NS + NS) (NH = NS/2;
// with NS < 8 the first half takes all of them)
template <int CELL, int N, int KS>
__device__ void bwd_epilogue(const BRun& a, const BCtx& c, int row, int hf, uint32_t acc_base) {
  constexpr int G = CellInfo<CELL>::G;
  constexpr int NS = N / KS;
  constexpr int NC4 = NS / 4;
  constexpr int ACC = N < 32 ? 32 : N;
  constexpr bool TWO = NS >= 8;          // both halves take columns
  constexpr int NH = TWO ? NS / 2 : NS;  // columns of a half
  constexpr int NL = NH < 16 ? NH : 16;  // columns per TMEM load
  const StackBwdLayer& ly = a.ly;
  const int T = a.T, B = a.B, H = a.H, GH = G * H, u = a.u_pack;
  const int me = c.me;
  const int j = c.ub * kUnits + row;
  const int lane = threadIdx.x & 31;
  const uint32_t lane_q = static_cast<uint32_t>(row & ~31) << 16;
  int prow[G];
#pragma unroll
  for (int g = 0; g < G; ++g) prow[g] = packed_row(g, j, G, u);
  float4* rbuf = reinterpret_cast<float4*>(c.smem + a.sm.rbuf);
  auto rb_at = [&](int p, int s, int ch) -> float4* { return rbuf + ((p * (KS - 1) + s) * NC4 + ch) * 128; };
  const bool act = TWO || hf == 0;  // this half takes columns
  const int c0h = hf * NH;          // first slice column of this half
  const int b0 = me * NS + c0h;     // its first batch entry
  const int nval = act ? min(NH, B - b0) : 0;
  // carried state: LSTM dc flowing into step s, GRU dh_{s+1} z_{s+1}
  float carry[NH];
#pragma unroll
  for (int cc = 0; cc < NH; ++cc)
    carry[cc] = (CELL == LSTM && ly.dcT && cc < nval) ? ly.dcT[(size_t)(b0 + cc) * H + j] : 0.f;

  for (int ti = 0; ti <= T; ++ti) {
    const int s = T - 1 - ti;  // reverse step; -1: dh0 = dGh_0 W_h
    const int acc = ti & 1, par = ti & 1;
    const uint32_t ph = (uint32_t)(ti >> 1) & 1u;
    if (KS > 1 && threadIdx.x == 64) tc::mbar_arrive_expect_tx(&c.rbar[par], (uint32_t)((KS - 1) * 128 * NS * 4));
    // ---- inputs of the pointwise step, independent of the recurrence: only
    // loads here, every conversion after the accumulator wait, so that all
    // columns' loads are in flight together (a conversion per column made
    // each column's load complete before the next one was issued).
    // Addresses are clamped into range instead of predicating the loads (a
    // value selected against 0 right after its load is consumed there):
    // columns past the batch are never stored, step -1 runs no pointwise
    // step, and c_{-1} without c0 is zeroed where it is used.
    float gv[G][NH], cs[NH], cp[NH], hnv[NH];
    unsigned short hpr[NH];
    uint32_t dyr[NH];  // the gradient from above as stored: bf16 bits, or float bits with dy_f32
    const int sl = s < 0 ? 0 : s;
    const bool cp_zero = CELL == LSTM && sl == 0 && !ly.c0;
#pragma unroll
    for (int cc = 0; cc < NH; ++cc) {
      const int b = min(b0 + cc, B - 1);
      const size_t bs = (size_t)sl * B + b;
#pragma unroll
      for (int g = 0; g < G; ++g) gv[g][cc] = ly.gates[bs * GH + prow[g]];
      if constexpr (CELL == LSTM) {
        cs[cc] = ly.c[bs * H + j];
        const float* cpp = sl > 0 ? ly.c + (bs - B) * H + j : (ly.c0 ? ly.c0 + (size_t)b * H + j : ly.c + bs * H + j);
        cp[cc] = *cpp;
      } else if constexpr (CELL == GRU) {
        hnv[cc] = ly.hn[bs * H + j];
        hpr[cc] = reinterpret_cast<const unsigned short*>(ly.hseq)[bs * H + j];  // slot s holds h_{s-1}
      }
    }
    // (one loop per storage type: the branch stays outside the loads)
    if (!ly.dy) {
#pragma unroll
      for (int cc = 0; cc < NH; ++cc) dyr[cc] = 0u;
    } else if (ly.dy_f32) {
      const uint32_t* dp = reinterpret_cast<const uint32_t*>(ly.dy) + (size_t)sl * B * H + j;
#pragma unroll
      for (int cc = 0; cc < NH; ++cc) dyr[cc] = dp[(size_t)min(b0 + cc, B - 1) * H];
    } else {
      const unsigned short* dp = reinterpret_cast<const unsigned short*>(ly.dy) + (size_t)sl * B * H + j;
#pragma unroll
      for (int cc = 0; cc < NH; ++cc) dyr[cc] = dp[(size_t)min(b0 + cc, B - 1) * H];
    }
    // ---- accumulator of this step: this half's columns of every chunk's
    // slice, its own summed, the others sent to their owners
    float sum[NH];
#pragma unroll
    for (int cc = 0; cc < NH; ++cc) sum[cc] = 0.f;
    bool ok;
    {
      int w = 1;
      if (lane == 0) w = tc::mbar_wait(&c.tfull[acc], ph, c.abort_flag, a.err, a.limit_ns) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, w, 0) != 0;
    }
    if (ok) {
      tc::fence_after_sync();
      if (act) {
#pragma unroll
        for (int p = 0; p < KS; ++p) {
#pragma unroll
          for (int l0 = 0; l0 < NH; l0 += NL) {
            float w[NL];
            tc::tmem_load_cols<NL>(c.tmem + lane_q + acc_base + (uint32_t)(acc * ACC + p * NS + c0h + l0), w);
            if (p == me) {
#pragma unroll
              for (int q = 0; q < NL; ++q) sum[l0 + q] += w[q];
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
      abort_cluster(c.abort_flag, a.cluster);
    }
    tc::named_bar(1, 256);
    if (*reinterpret_cast<volatile int*>(c.ep_fail)) break;
    if (act) {
#pragma unroll
      for (int k = 0; k < KS; ++k) {
        if (k == me) continue;
        const int slot = k < me ? k : k - 1;
#pragma unroll
        for (int q4 = 0; q4 < NH / 4; ++q4) {
          const float4 q = rb_at(par, slot, c0h / 4 + q4)[row];
          sum[4 * q4] += q.x;
          sum[4 * q4 + 1] += q.y;
          sum[4 * q4 + 2] += q.z;
          sum[4 * q4 + 3] += q.w;
        }
      }
    }
    if (s < 0) {
      // ---- dh0 (GRU: plus the carried dh_0 z_0) and dc0
#pragma unroll
      for (int cc = 0; cc < NH; ++cc) {
        if (cc >= nval) break;
        const size_t bj = (size_t)(b0 + cc) * H + j;
        if (ly.dh0) ly.dh0[bj] = __float2bfloat16_rn(sum[cc] + (CELL == GRU ? carry[cc] : 0.f));
        if (CELL == LSTM && ly.dc0) ly.dc0[bj] = carry[cc];
      }
      break;
    }
    // ---- pointwise step s: the gate gradients of this unit and batch slice
    float dgx[G][NH], dgh[G][NH], dyv[NH], hp[NH];
#pragma unroll
    for (int cc = 0; cc < NH; ++cc) {
      dyv[cc] = __uint_as_float(ly.dy_f32 ? dyr[cc] : dyr[cc] << 16);
      // the gradient reaching the final state, at the first reverse step only
      if (s == T - 1 && ly.dhT && cc < nval) dyv[cc] += __bfloat162float(ly.dhT[(size_t)(b0 + cc) * H + j]);
      hp[cc] = __uint_as_float((uint32_t)hpr[cc] << 16);
    }
#pragma unroll
    for (int cc = 0; cc < NH; ++cc) {
      if constexpr (CELL == LSTM) {
        const float ig = gv[0][cc], fg = gv[1][cc], gg = gv[2][cc], og = gv[3][cc];
        const float d = sum[cc] + dyv[cc];
        const float tau = tanh_hw(cs[cc]);
        const float dcv = carry[cc] + d * og * (1.f - tau * tau);
        dgx[0][cc] = dcv * gg * ig * (1.f - ig);
        dgx[1][cc] = dcv * (cp_zero ? 0.f : cp[cc]) * fg * (1.f - fg);
        dgx[2][cc] = dcv * ig * (1.f - gg * gg);
        dgx[3][cc] = d * tau * og * (1.f - og);
        carry[cc] = dcv * fg;
      } else if constexpr (CELL == GRU) {
        const float r = gv[0][cc], z = gv[1][cc], n = gv[2][cc];
        const float d = sum[cc] + dyv[cc] + carry[cc];
        const float dan = d * (1.f - z) * (1.f - n * n);
        dgx[0][cc] = dan * hnv[cc] * r * (1.f - r);
        dgx[1][cc] = d * (hp[cc] - n) * z * (1.f - z);
        dgx[2][cc] = dan;
        dgh[0][cc] = dgx[0][cc];
        dgh[1][cc] = dgx[1][cc];
        dgh[2][cc] = dan * r;
        carry[cc] = d * z;
      } else {
        dgx[0][cc] = (sum[cc] + dyv[cc]) * simple_slope<CELL>(gv[0][cc]);
      }
    }
    // ---- stores, then publish step s of this layer
    const size_t base = ((size_t)s * B + b0) * GH;
#pragma unroll
    for (int cc = 0; cc < NH; ++cc) {
      if (cc >= nval) break;
      __nv_bfloat16* gx = ly.dgx + base + (size_t)cc * GH;
      if (CELL == LSTM && u == 1) {
        uint2 v;
        v.x = pack_bf16x2(dgx[0][cc], dgx[1][cc]);
        v.y = pack_bf16x2(dgx[2][cc], dgx[G - 1][cc]);
        *reinterpret_cast<uint2*>(gx + prow[0]) = v;
      } else {
#pragma unroll
        for (int g = 0; g < G; ++g) gx[prow[g]] = __float2bfloat16_rn(dgx[g][cc]);
      }
      if constexpr (CELL == GRU) {
        __nv_bfloat16* gh = ly.dgh + base + (size_t)cc * GH;
#pragma unroll
        for (int g = 0; g < G; ++g) gh[prow[g]] = __float2bfloat16_rn(dgh[g][cc]);
      }
    }
    tc::fence_proxy_async_global();
    tc::named_bar(1, 256);
    if (threadIdx.x == 64 && !(a.test_skip_publish && blockIdx.x == 0 && ti == 0))
      red_release_add_u32(a.cnt + (size_t)c.li * T + s, 1u);
  }
}

// SA: some chunk keeps weights in shared memory (a separate variant: the
// extra MMA loop slowed the issue of the TMEM-only products by ~5% measured)
template <int CELL, int N, bool SA>
__global__ void __launch_bounds__(kThreads, 1)
    stack_bwd_kernel(const __grid_constant__ BwdMaps maps, const __grid_constant__ StackBwdArgs p) {
  constexpr int RING = N * 128;
  constexpr uint32_t TMEM_COLS = 512;  // weights (kc / 2 columns) + two accumulators
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
  BRun a;
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
  a.want_own = (unsigned)p.ctas[li];
  a.want_above = li + 1 < p.nl ? (unsigned)p.ctas[li + 1] : 0u;
  a.sm = p.sm;
  a.ly = p.lay[li];
  const int NB = a.sm.stages;
  BCtx c;
  c.smem = smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + a.sm.bars);
  c.full = bars;
  c.empty = c.full + kBufs;
  c.tfull = c.empty + kBufs;
  c.tempty = c.tfull + 2;
  c.rbar = c.tempty + 2;
  c.abar = c.rbar + 2;
  c.dbar = c.abar + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(c.dbar + 1);
  c.abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  c.ep_fail = reinterpret_cast<int*>(tmem_slot + 2);
  c.li = li;
  c.ks = p.ks[li];
  c.kr = p.kr[li];
  const int local = (int)blockIdx.x - p.cta0[li];
  c.ub = local / c.ks;
  c.me = local % c.ks;
  c.crank = a.cluster > 1 ? (int)tc::cluster_ctarank() : 0;
  const StackBwdLayer& ly = a.ly;
  const bool rec = c.me < c.kr;  // chunk of the recurrent part (else from above)
  const int k0 = (rec ? c.me : c.me - c.kr) * a.kc;
  const int nkb = a.kc / 64;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NB; ++i) {
      tc::mbar_init(c.full + i, 1);
      tc::mbar_init(c.empty + i, 1);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(c.tfull + i, 1);
      tc::mbar_init(c.tempty + i, 8);
      tc::mbar_init(c.rbar + i, 1);
    }
    tc::mbar_init(c.abar, 8);
    tc::mbar_init(c.dbar, 1);
    *c.abort_flag = 0;
    *c.ep_fail = 0;
    tc::fence_mbar_init();
    tc::tma_prefetch_desc(rec ? &maps.rec[li] : &maps.above[li]);
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, TMEM_COLS);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (a.cluster > 1) tc::cluster_sync_all();
  c.tmem = *tmem_slot;
  // TMEM columns [0, kct/2): the chunk's weights (k past kct in shared memory); then the accumulators
  const uint32_t acc_base = (uint32_t)(a.kct / 2);

  int last_par[kBufs];
  for (int i = 0; i < kBufs; ++i) last_par[i] = -1;
  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t buf = 0, phase = 0;
      const CUtensorMap* src = rec ? &maps.rec[li] : &maps.above[li];
      for (int ti = 0; ti <= a.T; ++ti) {
        const int s = a.T - 1 - ti;
        bool ok = true;
        if (rec) {
          if (s < a.T - 1)
            ok = wait_count(a.cnt + (size_t)li * a.T + s + 1, a.want_own, c.abort_flag, a.cluster, a.err, a.limit_ns);
        } else if (s >= 0 && ly.wait_above) {
          ok = wait_count(a.cnt + (size_t)(li + 1) * a.T + s, a.want_above, c.abort_flag, a.cluster, a.err,
                          a.limit_ns);
        }
        if (!ok) break;
        tc::fence_proxy_async_global();
        // recurrent: dGh_{s+1} (past the end at s = T-1: zeros); above: dGx^{l+1}_s
        // (before the start at s = -1: zeros)
        const int slot = rec ? s + 1 : s;
        if (!tc::mbar_wait(c.empty + buf, phase ^ 1, c.abort_flag, a.err, a.limit_ns)) break;
        tc::mbar_arrive_expect_tx(c.full + buf, (uint32_t)(nkb * RING));
        last_par[buf] = (int)phase;
        tc::tma_load_3d(smem + a.sm.ring + buf * nkb * RING, src, c.full + buf, 0, slot * a.B, k0 / 64);
        if (++buf == (uint32_t)NB) {
          buf = 0;
          phase ^= 1;
        }
      }
      if (*c.abort_flag) abort_cluster(c.abort_flag, a.cluster);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = tc::idesc_bf16(128, N, 0, 0);
      const int nkt = a.kct / 64;
      const uint64_t ad0 = tc::sdesc_sw128(tc::smem_addr(smem + a.sm.a), 16, 1024);
      bool ok = tc::mbar_wait(c.abar, 0, c.abort_flag, a.err, a.limit_ns);
      tc::fence_after_sync();
      uint32_t buf = 0, phase = 0;
      for (int ti = 0; ti <= a.T && ok; ++ti) {
        const int acc = ti & 1;
        if (!tc::mbar_wait(c.tempty + acc, ((uint32_t)(ti >> 1) & 1u) ^ 1u, c.abort_flag, a.err, a.limit_ns)) break;
        tc::fence_after_sync();
        const uint32_t d = c.tmem + acc_base + (uint32_t)(acc * (N < 32 ? 32 : N));
        if (!tc::mbar_wait(c.full + buf, phase, c.abort_flag, a.err, a.limit_ns)) break;
        tc::fence_after_sync();
        const uint32_t sb0 = tc::smem_addr(smem + a.sm.ring + buf * nkb * RING);
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
        if constexpr (SA) {
          // the k blocks past kct: A from the swizzled blocks in shared memory
          for (int i = 0; i < 4 * (nkb - nkt); ++i) {
            const int kb = nkt + (i >> 2), kk = i & 3;
            tc::mma_bf16(d, ad0 + (uint64_t)(((i >> 2) * 16384 + kk * 32) >> 4),
                         bd0 + (uint64_t)((kb * RING + kk * 32) >> 4), idesc, 1u);
          }
        } else {
          (void)ad0;
        }
        tc::mma_commit(c.empty + buf);
        if (++buf == (uint32_t)NB) {
          buf = 0;
          phase ^= 1;
        }
        tc::mma_commit(c.tfull + acc);
      }
      tc::mma_commit(c.dbar);
      const uint64_t t0 = globaltimer_ns();
      while (!tc::mbar_try_wait(c.dbar, 0) && globaltimer_ns() - t0 < 1000000ull) {
      }
      if (*c.abort_flag) abort_cluster(c.abort_flag, a.cluster);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int row = (warp & 3) * 32 + lane;
    const int hf = (warp - 2) >> 2;  // half of the epilogue (two warps per TMEM lane quadrant)
    {
      // this unit's column of the chunk's weights into TMEM: A[j][k] =
      // W[k0 + k][j], two consecutive k per 32-bit column; the two halves
      // take alternate 32-wide k blocks
      const int j = c.ub * kUnits + row;
      const unsigned short* wcol =
          reinterpret_cast<const unsigned short*>(rec ? ly.Wh : ly.Wx_above) + (size_t)k0 * a.H + j;
      const uint32_t lane_q = static_cast<uint32_t>(row & ~31) << 16;
      for (int c16 = hf; c16 < a.kct / 32; c16 += 2) {
        float v[16];
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          const size_t k = (size_t)(c16 * 32 + 2 * q);
          const uint32_t lo = wcol[k * a.H], hi = wcol[(k + 1) * a.H];
          v[q] = __uint_as_float(lo | (hi << 16));
        }
        tc::tmem_store16(c.tmem + lane_q + (uint32_t)(c16 * 16), v);
      }
      // k past kct into shared memory as K-major 128 x 64 blocks with the
      // 128-byte swizzle (16-byte piece q of row r at piece q ^ (r % 8))
      if constexpr (SA) {
        for (int q8 = hf; q8 < (a.kc - a.kct) / 8; q8 += 2) {
          uint32_t w[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const size_t k = (size_t)(a.kct + 8 * q8 + 2 * i);
            w[i] = (uint32_t)wcol[k * a.H] | ((uint32_t)wcol[(k + 1) * a.H] << 16);
          }
          const int blk = q8 >> 3, q = q8 & 7;
          *reinterpret_cast<uint4*>(smem + a.sm.a + blk * 16384 + row * 128 + ((q ^ (row & 7)) << 4)) =
              make_uint4(w[0], w[1], w[2], w[3]);
        }
        tc::fence_proxy_async_smem();  // generic stores read by the tensor core (async proxy)
      }
      tc::tmem_store_wait();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(c.abar);
    }
    // the geometry keeps 4..16 batch columns per CTA: only those variants exist
    if constexpr (N / 2 <= 16) {
      if (c.ks == 2) bwd_epilogue<CELL, N, 2>(a, c, row, hf, acc_base);
    }
    if (c.ks == 4) bwd_epilogue<CELL, N, 4>(a, c, row, hf, acc_base);
    if constexpr (N / 8 >= 4) {
      if (c.ks == 8) bwd_epilogue<CELL, N, 8>(a, c, row, hf, acc_base);
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0 && lane == 0 && *c.abort_flag) {
    for (int i = 0; i < NB; ++i) {
      if (last_par[i] < 0) continue;
      const uint64_t t0 = globaltimer_ns();
      while (!tc::mbar_try_wait(c.full + i, (uint32_t)last_par[i]) && globaltimer_ns() - t0 < 1000000ull) {
      }
    }
  }
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(c.tmem, TMEM_COLS);
  }
  if (a.cluster > 1) tc::cluster_sync_all();
}

// Geometry of a backward launch over layers [0, nl) of a group (lay[0] the
// lowest): per layer the K chunk width kc (a multiple of 64 dividing G*H),
// the chunks of the recurrent part (kr = G*H / kc) and in all (ks = kr, or
// 2 kr with a layer above), the CTAs (H / 128 unit blocks x ks).  A CTA
// reduces N / ks batch columns (4..16); chunks are narrowed on the layers
// with the fewest while the CTAs stay within `budget`, as in the forward.
struct BGeom {
  int N, cluster, ctas, sa;  // sa: some chunk keeps weights in shared memory
  int kc[kStackMaxLayers], kct[kStackMaxLayers], kr[kStackMaxLayers], ks[kStackMaxLayers],
      cta0[kStackMaxLayers + 1], lctas[kStackMaxLayers];
  BSmem sm;
};

int bwd_geometry(int cell, int H, int B, int nl, int has_top, int budget, BGeom* g) {
  if (nl < 1 || nl > kStackMaxLayers || B < 1 || B > 64 || H % kUnits) return RNN_ERR_UNSUPPORTED;
  const int G = cell == LSTM ? 4 : cell == GRU ? 3 : 1;
  const int GH = G * H;
  // at least 32 batch columns: eight K chunks then still leave each CTA 4
  // columns of the reduction (the columns past the batch compute on zeros)
  g->N = B <= 32 ? 32 : 64;
  const int acc_cols = 2 * (g->N < 32 ? 32 : g->N);
  const int kt_max = 2 * (512 - acc_cols);  // k that fit TMEM beside the two accumulators
  constexpr int kKs = 256;                  // at most this many k of a chunk in shared memory
  auto valid = [&](int l, int kc) {
    if (kc % 64 || GH % kc || kc > kt_max + kKs) return false;
    const int parts = (has_top && l == nl - 1) ? 1 : 2;
    const int ks = parts * (GH / kc);
    return (ks == 2 || ks == 4 || ks == 8) && g->N / ks >= 4 && g->N / ks <= 16;
  };
  auto set = [&](int l, int kc) {
    g->kc[l] = kc;
    g->kct[l] = std::min(kc, kt_max / 64 * 64);
    g->kr[l] = GH / kc;
    g->ks[l] = ((has_top && l == nl - 1) ? 1 : 2) * g->kr[l];
  };
  const int rbs = H / kUnits;
  int cta = 0;
  for (int l = 0; l < nl; ++l) {
    // the widest chunk of at most 512, else the narrowest wider one
    int kc = 0;
    for (int c = 512; c >= 64 && !kc; c -= 64)
      if (valid(l, c)) kc = c;
    for (int c = 576; c <= kt_max + kKs && !kc; c += 64)
      if (valid(l, c)) kc = c;
    if (!kc) return RNN_ERR_UNSUPPORTED;
    set(l, kc);
    cta += rbs * g->ks[l];
  }
  // over the budget: widen (kc -> 2 kc, halving ks) the layer with the most
  // chunks that can be widened, while any can
  while (cta > budget) {
    int lw = -1;
    for (int l = 0; l < nl; ++l)
      if (valid(l, 2 * g->kc[l]) && (lw < 0 || g->ks[l] > g->ks[lw])) lw = l;
    if (lw < 0) break;
    cta -= rbs * g->ks[lw];
    set(lw, 2 * g->kc[lw]);
    cta += rbs * g->ks[lw];
  }
  // narrow the layers with the fewest chunks (kc -> kc / 2, doubling ks)
  for (;;) {
    int kmin = 16;
    for (int l = 0; l < nl; ++l) kmin = std::min(kmin, g->ks[l]);
    int extra = 0;
    bool can = true;
    for (int l = 0; l < nl; ++l) {
      if (g->ks[l] != kmin) continue;
      if (!valid(l, g->kc[l] / 2)) can = false;
      extra += rbs * g->ks[l];
    }
    if (!can || cta + extra > budget) break;
    for (int l = 0; l < nl; ++l)
      if (g->ks[l] == kmin) set(l, g->kc[l] / 2);
    cta += extra;
  }
  int ksmax = 1, kcmax = 0, kcsmax = 0;
  cta = 0;
  for (int l = 0; l < nl; ++l) {
    ksmax = std::max(ksmax, g->ks[l]);
    kcmax = std::max(kcmax, g->kc[l]);
    kcsmax = std::max(kcsmax, g->kc[l] - g->kct[l]);
    g->sa = kcsmax > 0 ? 1 : 0;
    g->cta0[l] = cta;
    g->lctas[l] = rbs * g->ks[l];
    cta += g->lctas[l];
  }
  g->cta0[nl] = cta;
  g->ctas = cta;
  g->cluster = ksmax;
  if (cta > budget) return RNN_ERR_LAUNCH;
  for (int l = 0; l < nl; ++l)
    if (g->lctas[l] % ksmax) return RNN_ERR_UNSUPPORTED;
  bool fit = false;
  for (int bufs : {2, 1}) {
    g->sm = bwd_layout(g->N, kcmax, ksmax, bufs, kcsmax);
    if (g->sm.total + 1024 <= 227 * 1024) {
      fit = true;
      break;
    }
  }
  return fit ? RNN_OK : RNN_ERR_UNSUPPORTED;
}

template <int CELL, int N, bool SA>
int launch_t(const Launch& L, const BwdMaps& maps, const StackBwdArgs& a, const BGeom& g, bool query_only,
             int num_sms) {
  auto k = stack_bwd_kernel<CELL, N, SA>;
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

int dispatch(const Launch& L, int cell, const BwdMaps& maps, const StackBwdArgs& a, const BGeom& g, bool query_only,
             int num_sms) {
  const bool sa = g.sa != 0;
  if (sa && g.N > 32) return RNN_ERR_UNSUPPORTED;  // the shared-memory chunks only fit up to 32 columns
#define RNN_S(C)                                                                                  \
  if (cell == C) {                                                                                \
    if (g.N == 16) return sa ? launch_t<C, 16, true>(L, maps, a, g, query_only, num_sms)          \
                             : launch_t<C, 16, false>(L, maps, a, g, query_only, num_sms);        \
    if (g.N == 32) return sa ? launch_t<C, 32, true>(L, maps, a, g, query_only, num_sms)          \
                             : launch_t<C, 32, false>(L, maps, a, g, query_only, num_sms);        \
    return launch_t<C, 64, false>(L, maps, a, g, query_only, num_sms);                            \
  }
  RNN_S(LSTM) RNN_S(GRU) RNN_S(TANH) RNN_S(RELU)
#undef RNN_S
  return RNN_ERR_UNSUPPORTED;
}

}  // namespace

int stack_bwd_check(int cell, int H, int B, int nl, int has_top, int u_pack, int num_sms, int* ctas, int* budget) {
  if (u_pack < 1) return RNN_ERR_UNSUPPORTED;
  // the widest geometry whose clusters all co-reside: narrowing chunks adds
  // CTAs, and clusters of 8 may not all fit even where the CTAs do
  int b = num_sms > 0 ? num_sms : 152;
  for (;;) {
    BGeom g;
    RNN_TRY_LOCAL(bwd_geometry(cell, H, B, nl, has_top, b, &g));
    int rc = RNN_OK;
    if (num_sms > 0) {
      BwdMaps maps{};
      StackBwdArgs a{};
      Launch L{};
      rc = dispatch(L, cell, maps, a, g, true, num_sms);
    } else if (g.cluster == 8 && g.ctas > 14 * 8) {
      rc = RNN_ERR_LAUNCH;  // host-side planning: GB300 held 14 clusters of 8 of this kernel at once, not 16
    }
    if (rc == RNN_OK) {
      if (ctas) *ctas = g.ctas;
      if (budget) *budget = b;
      return RNN_OK;
    }
    if (rc != RNN_ERR_LAUNCH) return rc;
    b = g.ctas - 1;  // a geometry with fewer CTAs, if there is one
  }
}

int stack_bwd(const Launch& L, int cell, const StackBwdArgs& in) {
  BGeom g;
  const int has_top = in.lay[in.nl - 1].Wx_above == nullptr ? 1 : 0;
  RNN_TRY_LOCAL(bwd_geometry(cell, in.H, in.B, in.nl, has_top, in.budget, &g));
  const int G = cell == LSTM ? 4 : cell == GRU ? 3 : 1;
  const int GH = G * in.H;
  StackBwdArgs a = in;
  a.cluster = g.cluster;
  for (int l = 0; l < in.nl; ++l) {
    a.kcl[l] = g.kc[l];
    a.kctl[l] = g.kct[l];
    a.kr[l] = g.kr[l];
    a.ks[l] = g.ks[l];
    a.cta0[l] = g.cta0[l];
    a.ctas[l] = g.lctas[l];
  }
  a.cta0[in.nl] = g.cta0[in.nl];
  a.sm.stages = g.sm.bufs;
  a.sm.a = g.sm.a;
  a.sm.ring = g.sm.ring;
  a.sm.rbuf = g.sm.rbuf;
  a.sm.smg = 0;
  a.sm.smhn = 0;
  a.sm.bars = g.sm.bars;
  BwdMaps maps;
  memset(&maps, 0, sizeof(maps));
  const long long rows = (long long)in.T * in.B;
  for (int l = 0; l < in.nl; ++l) {
    const StackBwdLayer& ly = in.lay[l];
    const bool top = has_top && l == in.nl - 1;
    if (!ly.Wh || !ly.dgx || !ly.dgh || !ly.gates || (reinterpret_cast<uintptr_t>(ly.Wh) & 15))
      return RNN_ERR_INVALID_ARG;
    if (cell == LSTM && !ly.c) return RNN_ERR_INVALID_ARG;
    if (cell == GRU && (!ly.hn || !ly.hseq)) return RNN_ERR_INVALID_ARG;
    if (top != (ly.Wx_above == nullptr) || top != (ly.dgx_above == nullptr)) return RNN_ERR_INVALID_ARG;
    if ((l + 1 < in.nl) != (ly.wait_above != 0)) return RNN_ERR_INVALID_ARG;  // counters of layers in this launch only
    RNN_TRY_LOCAL(encode_seq3(&maps.rec[l], ly.dgh, rows, GH, g.N, g.kc[l] / 64));
    if (!top) RNN_TRY_LOCAL(encode_seq3(&maps.above[l], ly.dgx_above, rows, GH, g.N, g.kc[l] / 64));
  }
  return dispatch(L, cell, maps, a, g, false, L.num_sms);
}

}  // namespace rnn
