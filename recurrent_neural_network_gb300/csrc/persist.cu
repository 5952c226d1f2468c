// persist.cu -- persistent forward recurrence for small batches.
//
// "Persistent RNNs: Stashing Recurrent Weights On-Chip" (citing snippets on
// its page): cache the recurrent weights on-chip across timesteps and run all
// timesteps in one kernel launch; small-batch RNNs are matrix-vector work.
// Each CTA owns uc hidden units (all G gates of them) and keeps their rows of
// the packed W_h in registers as mma.sync A fragments for the whole sequence.
// Per timestep it reads h_{t-1} (all B x H values) from global memory, forms
// its G*uc x B slice of h_{t-1} W_h^T on the tensor cores (split over K
// across 8 warps, reduced through shared memory), applies the cell update to
// its units and publishes its part of h_t.  Time may also run backwards
// (the reverse direction of a bidirectional layer).
//
// Step hand-off, two variants.
//
// Cluster exchange (default where clusters of 2-8 CTAs co-reside): each CTA
// writes its slice of h_t as tagged 8-byte words (two bf16 values and the
// step number + 1) into a global ping-pong buffer; a word carries its own
// validity, so the producer needs no release fence.  The CTAs of a cluster
// split the words of h_{t-1} among them: each polls its share until the tags
// match, scatters the values into the h_{t-1} buffer in the shared memory of
// every CTA of the cluster, and one cluster barrier later every CTA holds
// all of h_{t-1} on chip.  Each word is polled by one CTA per cluster, not by
// every CTA, which keeps the polling off the L2 slices' critical path.
//
// Counter (fallback): after its h_t stores a CTA makes one release arrival on
// the step's counter (one counter per timestep, zeroed before the launch);
// one thread per CTA polls the counter of the previous step until every CTA
// has arrived, then the CTA reads h_{t-1} once through L2.
//
// fp8 stash (PersistArgs::Wh8 set): W_h is held as e4m3 bytes with one fp32
// scale per packed row, in shared memory (in fragment order, read once per
// step), so that LSTM and GRU layers twice as wide as the register-resident
// bf16 variant keep their recurrent weights on chip ("Persistent RNNs" page,
// citing snippets: on-chip storage is small and inflexible in precision).
// Each step widens the bytes to f16 with an exact bit rearrangement, runs the
// product as f16 MMAs against h (bf16 converted to f16) and applies the row
// scales to the fp32 sums.
//
// The cluster variant first checks that its launch has the cluster size the
// arguments name (it addresses every peer's shared memory); otherwise every
// CTA records DEV_BAD_CLUSTER and returns.
//
// Every wait is bounded (globaltimer); on timeout the CTA records
// DEV_TIMEOUT_STEP in the error word and leaves (in the cluster variant the
// whole cluster leaves together, after the step's cluster barrier).
// Co-residency of all CTAs is guaranteed by a cooperative launch.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "../../include/rnn.h"
#include "common.cuh"
#include "launchers.h"
#include "tc.cuh"

namespace rnn {

namespace {

__device__ __forceinline__ void mma_bf16_16816(float* d, const uint32_t* a, const uint32_t* b) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

__device__ __forceinline__ void mma_f16_16816(float* d, const uint32_t* a, const uint32_t* b) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// Two e4m3 bytes of x (bytes 0,1 with sel 0x1404, bytes 2,3 with sel 0x3424)
// as an f16 pair worth 2^-8 times their value.  Each byte s.eeee.mmm lands in
// the high byte of a half (sign at bit 15), and the seven bits below the sign
// move down one place, giving exponent field 0eeee and mantissa mmm0000000:
// 2^(e-15) (1 + m/8) for normal bytes and 2^-14 (m/8) for subnormal ones,
// i.e. the e4m3 value (bias 7) times 2^-8, exactly.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2_lo8(uint32_t x, uint32_t sel) {
  const uint32_t p = __byte_perm(x, 0u, sel);
  return ((p >> 1) & 0x3F803F80u) | (p & 0x80008000u);
}
// bf16 pair -> f16 pair (round to nearest)
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t u) {
  const __half2 h = __floats2half2_rn(__uint_as_float(u << 16), __uint_as_float(u & 0xFFFF0000u));
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ unsigned int ld_acquire(const unsigned int* p) {
  unsigned int v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
// Release-ordered add: this thread's earlier writes, and those it has
// synchronised with through a barrier, are visible before the count changes.
__device__ __forceinline__ void red_release_add(unsigned int* p, unsigned int v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint64_t ld_relaxed_u64(const uint64_t* p) {
  uint64_t v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_relaxed_u64(uint64_t* p, uint64_t v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ void st_dsmem_u32(uint32_t cluster_addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}
// Asynchronous 4-byte store into the shared memory of a CTA of the cluster
// whose completion is counted (4 transaction bytes) on that CTA's mbarrier.
__device__ __forceinline__ void st_async_u32(uint32_t cluster_addr, uint32_t v, uint32_t cluster_bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(cluster_addr),
               "r"(v), "r"(cluster_bar)
               : "memory");
}
// every thread of every CTA of the cluster (threads may arrive diverged)
__device__ __forceinline__ void cluster_barrier() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

__device__ __forceinline__ unsigned short bf16_bits(float v) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(v));
}

// most tagged words one thread polls per step (the cluster size is chosen so
// that B*H/2 words over the cluster's CTAs' threads stay within it)
constexpr int kMaxWords = 4;

// NT threads (8 or 16 warps, each taking KT 16-deep k-tiles of W_h's K range).
// HO: hand-off of h_t.  0 counters; 1 tagged words gathered per cluster, then a
// cluster barrier; 2 tagged words gathered per cluster with asynchronous
// stores into every peer, each CTA waiting on its own mbarrier for the bytes
// of its copy of h_{t-1} (no barrier across the cluster per step).
template <int CELL, int MT, int KT, int HO, bool W8, int NT>
__global__ void __launch_bounds__(NT, 1) persist_fwd_kernel(const PersistArgs a) {
  constexpr bool XCL = HO > 0;
  constexpr int G = CellInfo<CELL>::G;
  constexpr int ROWS = MT * 16;  // = G * uc
  constexpr int NWARP = NT / 32;
  __shared__ float part[NWARP][ROWS][8];
  __shared__ float sums[ROWS][8];
  __shared__ float rscale[W8 ? ROWS : 1];  // fp8 stash: row scale x 2^8
  __shared__ int abort_flag;
  __shared__ int abort_x[2];  // cluster exchange: set in every CTA of the cluster by one that gave up
  __shared__ __align__(8) uint64_t hbar[2];  // HO = 2: bytes of h_{t-1} landed in buffer t & 1
  // dynamic shared memory: fp8 stash of this CTA's W_h rows (ROWS x H bytes
  // in fragment order), then for the cluster exchange the h_{t-1} ping-pong
  // [2][B][H + 8] bf16 (rows padded so that the eight batch rows of a
  // fragment load fall in distinct banks)
  extern __shared__ __align__(16) unsigned char dsm[];
  uint32_t* w8s = reinterpret_cast<uint32_t*>(dsm);
  unsigned char* hbuf = dsm + (W8 ? ROWS * a.H : 0);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int uc = ROWS / G;
  const int H = a.H, B = a.B, GH = G * H;
  const int jbase = blockIdx.x * uc;
  // time order: step t runs time t (forward) or T-1-t (reverse); the h
  // sequence keeps h(time) at slot time+1 forward, at slot time in reverse,
  // and the initial state at slot 0 or T
  const int slot_h0 = a.reverse ? a.T : 0;
  if (threadIdx.x == 0) abort_flag = 0;

  // ---- this CTA's rows of W_h as A fragments (row r = g*uc + local unit),
  // in registers; fp8 stash: in shared memory, per row of a fragment the four
  // bytes at k, k+1, k+8, k+9, word i of (mt, kt) of this thread at
  // w8s[((warp * MT + mt) * KT + kt) * 64 + lane * 2 + i]
  uint32_t wf[W8 ? 1 : MT][W8 ? 1 : KT][4];
  {
    const int kw = warp * KT * 16;
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      const int r0 = mt * 16 + (lane >> 2), r1 = r0 + 8;
      const int p0 = packed_row(r0 / uc, jbase + r0 % uc, G, a.u_pack);
      const int p1 = packed_row(r1 / uc, jbase + r1 % uc, G, a.u_pack);
      if constexpr (W8) {
        const uint16_t* w0 = reinterpret_cast<const uint16_t*>(a.Wh8 + (size_t)p0 * H);
        const uint16_t* w1 = reinterpret_cast<const uint16_t*>(a.Wh8 + (size_t)p1 * H);
        for (int kt = 0; kt < KT; ++kt) {
          const int k = kw + kt * 16 + (lane & 3) * 2;
          uint32_t* d = w8s + ((warp * MT + mt) * KT + kt) * 64 + lane * 2;
          d[0] = (uint32_t)w0[k >> 1] | ((uint32_t)w0[(k + 8) >> 1] << 16);
          d[1] = (uint32_t)w1[k >> 1] | ((uint32_t)w1[(k + 8) >> 1] << 16);
        }
      } else {
        const uint32_t* w0 = reinterpret_cast<const uint32_t*>(a.Wh + (size_t)p0 * H);
        const uint32_t* w1 = reinterpret_cast<const uint32_t*>(a.Wh + (size_t)p1 * H);
#pragma unroll
        for (int kt = 0; kt < KT; ++kt) {
          const int k = kw + kt * 16 + (lane & 3) * 2;
          wf[mt][kt][0] = w0[k >> 1];
          wf[mt][kt][1] = w1[k >> 1];
          wf[mt][kt][2] = w0[(k + 8) >> 1];
          wf[mt][kt][3] = w1[(k + 8) >> 1];
        }
      }
    }
  }
  if constexpr (W8) {
    for (int r = threadIdx.x; r < ROWS; r += NT)
      rscale[r] = a.wscale[packed_row(r / uc, jbase + r % uc, G, a.u_pack)] * 256.f;
  }

  // ---- cell-update threads: one (unit, batch row) pair each
  const int q = threadIdx.x;
  const int jl = q % uc, bq = q / uc;
  const bool pair = bq < B && q < uc * 8;
  const int j = jbase + jl;
  float c_state = 0.f, h_prev = 0.f;
  int pcol[G];
#pragma unroll
  for (int g = 0; g < G; ++g) pcol[g] = packed_row(g, j, G, a.u_pack);
  if (pair) {
    if (CELL == LSTM && a.c0) c_state = a.c0[(size_t)bq * H + j];
    if (CELL == GRU) h_prev = __bfloat162float(a.hseq[((size_t)slot_h0 * B + bq) * H + j]);
  }
  const float bhn = (CELL == GRU && pair) ? a.bias_hn[j] : 0.f;
  const int HP2 = H / 2 + 4;            // words per padded h row
  const int NW = (H / 2) * B;           // tagged words of h per step
  const int WS = (uc * B) / 2;          // of which this CTA produces
  uint32_t crank = 0, csize = 1;
  // this thread's share of the tagged words of a step: w0 + NT i, i < nmine,
  // and where word i lands in an h buffer (word w of CTA c holds units jj,
  // jj+1 of batch row bq)
  int w0 = 0, nmine = 0;
  uint32_t offw[kMaxWords];
  if constexpr (XCL) {
    // the exchange addresses the shared memory of every CTA of the cluster:
    // a launch whose cluster is not the size the arguments promise leaves at
    // once (every CTA alike, before any peer access or cluster barrier)
    uint32_t ncta;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(ncta));
    if ((int)ncta != a.cluster || a.cluster < 2) {
      if (threadIdx.x == 0) raise_error(a.err, DEV_BAD_CLUSTER);
      return;
    }
    crank = tc::cluster_ctarank();
    csize = (uint32_t)a.cluster;
    const int per = NW / (int)csize;
    w0 = (int)crank * per + threadIdx.x;
    nmine = per > (int)threadIdx.x ? min(kMaxWords, (per - (int)threadIdx.x + NT - 1) / NT) : 0;
#pragma unroll
    for (int i = 0; i < kMaxWords; ++i) {
      const int w = w0 + i * NT;
      const int c = w / WS, q0 = 2 * (w - c * WS);
      const int bq = q0 / uc, jj = c * uc + (q0 - bq * uc);
      offw[i] = (uint32_t)(bq * HP2 * 4 + jj * 2);
    }
    const uint32_t* h0w = reinterpret_cast<const uint32_t*>(a.hseq + (size_t)slot_h0 * B * H);
    uint32_t* hw = reinterpret_cast<uint32_t*>(hbuf);
    for (int i = threadIdx.x; i < NW; i += NT) {
      const int b = i / (H / 2);
      hw[b * HP2 + (i - b * (H / 2))] = h0w[i];
    }
    if (threadIdx.x < 2) abort_x[threadIdx.x] = 0;
    if (HO == 2 && threadIdx.x == 0) {
      tc::mbar_init(&hbar[0], 1);
      tc::mbar_init(&hbar[1], 1);
      tc::fence_mbar_init();
    }
    // peers write into this CTA's buffers, barriers and flags only after this point
    cluster_barrier();
  }
  __syncthreads();

  const int nb = lane >> 2;  // batch column of this lane's B fragment
  const int kw = warp * KT * 16 + (lane & 3) * 2;
  for (int t = 0; t < a.T; ++t) {
    const int tm = a.reverse ? a.T - 1 - t : t;            // time of this step
    const int s_in = a.reverse ? a.T - t : t;              // slot of h before it
    const int s_out = a.reverse ? a.T - 1 - t : t + 1;     // slot of h after it
    // input projection of this step for the pair (independent of the recurrence)
    float pv[G];
    if (pair) {
      const float* prow = a.P + ((size_t)tm * B + bq) * GH;
#pragma unroll
      for (int g = 0; g < G; ++g) pv[g] = prow[pcol[g]];
    }
    // ---- wait until every CTA has published h_{t-1}, then load this warp's
    // B fragments of it
    if (XCL && t > 0) {
      // this CTA's share of the tagged words of h_{t-1}, scattered into
      // buffer t&1 of every CTA of the cluster
      const uint64_t* src = a.hx + (size_t)((t - 1) & 1) * NW;
      const uint32_t want = (uint32_t)t;
      const uint32_t hbase = tc::smem_addr(hbuf) + (uint32_t)((t & 1) * B * HP2 * 4);
      const uint32_t bar_local = tc::smem_addr(&hbar[t & 1]);
      // HO = 2: this CTA's buffer receives one 4-byte store per word from the
      // cluster's pollers (remote completions may come before this arrival)
      if (HO == 2 && threadIdx.x == 0) tc::mbar_arrive_expect_tx(&hbar[t & 1], (uint32_t)NW * 4u);
      // every round loads all of this thread's missing words at once, so a
      // word that is already there costs no extra round trip
      uint32_t pending = (1u << nmine) - 1u;
      bool bad = false;
      uint64_t t0 = 0;
      while (pending) {
        uint64_t v[kMaxWords];
#pragma unroll
        for (int i = 0; i < kMaxWords; ++i)
          if ((pending >> i) & 1u) v[i] = ld_relaxed_u64(src + w0 + i * NT);
#pragma unroll
        for (int i = 0; i < kMaxWords; ++i) {
          if (((pending >> i) & 1u) && (uint32_t)(v[i] >> 32) == want) {
            pending &= ~(1u << i);
            const uint32_t off = hbase + offw[i];
            if constexpr (HO == 2) {
              for (uint32_t r = 0; r < csize; ++r)
                st_async_u32(tc::mapa(off, r), (uint32_t)v[i], tc::mapa(bar_local, r));
            } else {
              for (uint32_t r = 0; r < csize; ++r) st_dsmem_u32(tc::mapa(off, r), (uint32_t)v[i]);
            }
          }
        }
        if (!pending) break;
        if (t0 == 0) {
          t0 = globaltimer_ns();
        } else if (globaltimer_ns() - t0 > a.limit_ns) {
          bad = true;
          break;
        }
      }
      if (bad) {
        raise_error(a.err, DEV_TIMEOUT_STEP);
        const uint32_t fo = tc::smem_addr(&abort_x[t & 1]);
        for (uint32_t r = 0; r < csize; ++r) st_dsmem_u32(tc::mapa(fo, r), 1u);
      }
      if constexpr (HO == 2) {
        // this CTA's copy of h_{t-1} is complete once all its bytes landed
        // (bounded; a peer that gave up marks abort_x here, and this CTA leaves)
        const uint32_t par = (uint32_t)((t - 1) >> 1) & 1u;
        bool ok = tc::mbar_try_wait_cluster(&hbar[t & 1], par);
        if (!ok) {
          const uint64_t w0t = globaltimer_ns();
          while (!(ok = tc::mbar_try_wait_cluster(&hbar[t & 1], par))) {
            if (*reinterpret_cast<volatile int*>(&abort_x[t & 1])) break;
            if (globaltimer_ns() - w0t > a.limit_ns) {
              raise_error(a.err, DEV_TIMEOUT_STEP);
              break;
            }
          }
        }
        if (!ok || bad) {
          // stop every CTA of the cluster at its next wait
          const uint32_t fo = tc::smem_addr(&abort_x[t & 1]);
          for (uint32_t r = 0; r < csize; ++r) st_dsmem_u32(tc::mapa(fo, r), 1u);
        }
        __syncthreads();
        if (*reinterpret_cast<volatile int*>(&abort_x[t & 1])) break;
      } else {
        cluster_barrier();
        if (*reinterpret_cast<volatile int*>(&abort_x[t & 1])) break;
      }
    }
    if (!XCL && t > 0) {
      if (threadIdx.x == 0) {
        const unsigned int* cnt = a.arrive + (t - 1);
        const unsigned int want = gridDim.x;
        if (ld_acquire(cnt) < want) {
          const uint64_t t0 = globaltimer_ns();
          while (ld_acquire(cnt) < want) {
            if (globaltimer_ns() - t0 > a.limit_ns) {
              abort_flag = 1;
              raise_error(a.err, DEV_TIMEOUT_STEP);
              break;
            }
          }
        }
      }
      __syncthreads();
      if (abort_flag) break;
    }
    // ---- partial products over this warp's K range (B fragments of h_{t-1}
    // from the cluster's shared-memory copy or through L2)
    float acc[MT][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;
    const uint32_t* hsx = reinterpret_cast<const uint32_t*>(hbuf) + ((t & 1) * B + nb) * HP2 + (kw >> 1);
    const uint32_t* hsg = reinterpret_cast<const uint32_t*>(a.hseq + ((size_t)s_in * B + min(nb, B - 1)) * H + kw);
    auto load_b = [&](int kt, uint32_t* b2) {
      if (nb >= B) {
        b2[0] = b2[1] = 0u;
      } else if (XCL) {
        b2[0] = hsx[kt * 8];
        b2[1] = hsx[kt * 8 + 4];
      } else {
        b2[0] = __ldcg(hsg + kt * 8);
        b2[1] = __ldcg(hsg + kt * 8 + 4);
      }
    };
    if constexpr (W8) {
#pragma unroll 4
      for (int kt = 0; kt < KT; ++kt) {
        uint32_t b2[2];
        load_b(kt, b2);
        const uint32_t hb[2] = {bf16x2_to_f16x2(b2[0]), bf16x2_to_f16x2(b2[1])};
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          const uint2 q = *reinterpret_cast<const uint2*>(w8s + ((warp * MT + mt) * KT + kt) * 64 + lane * 2);
          const uint32_t af[4] = {e4m3x2_to_f16x2_lo8(q.x, 0x1404u), e4m3x2_to_f16x2_lo8(q.y, 0x1404u),
                                  e4m3x2_to_f16x2_lo8(q.x, 0x3424u), e4m3x2_to_f16x2_lo8(q.y, 0x3424u)};
          mma_f16_16816(acc[mt], af, hb);
        }
      }
    } else {
      uint32_t bf[KT][2];
#pragma unroll
      for (int kt = 0; kt < KT; ++kt) load_b(kt, bf[kt]);
#pragma unroll
      for (int kt = 0; kt < KT; ++kt)
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) mma_bf16_16816(acc[mt], reinterpret_cast<const uint32_t*>(wf[mt][kt]), bf[kt]);
    }
    for (int mt = 0; mt < MT; ++mt) {
      const int r = mt * 16 + (lane >> 2), c = (lane & 3) * 2;
      part[warp][r][c] = acc[mt][0];
      part[warp][r][c + 1] = acc[mt][1];
      part[warp][r + 8][c] = acc[mt][2];
      part[warp][r + 8][c + 1] = acc[mt][3];
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < ROWS * 8; idx += NT) {
      const int r = idx >> 3, c = idx & 7;
      float s = 0.f;
#pragma unroll
      for (int w = 0; w < NWARP; ++w) s += part[w][r][c];
      if constexpr (W8) s *= rscale[r];
      sums[r][c] = s;
    }
    __syncthreads();
    // ---- cell update of this CTA's units
    uint32_t hv = 0;
    if (pair) {
      float av[G];
#pragma unroll
      for (int g = 0; g < G; ++g) av[g] = sums[g * uc + jl][bq];
      float hnew, gv[G];
      if constexpr (CELL == LSTM) {
        const float ig = sigm_hw(av[0] + pv[0]), fg = sigm_hw(av[1] + pv[1]);
        const float gg = tanh_hw(av[2] + pv[2]), og = sigm_hw(av[3] + pv[3]);
        c_state = fg * c_state + ig * gg;
        hnew = og * tanh_hw(c_state);
        gv[0] = ig; gv[1] = fg; gv[2] = gg; gv[G - 1] = og;
      } else if constexpr (CELL == GRU) {
        const float r = sigm_hw(av[0] + pv[0]), z = sigm_hw(av[1] + pv[1]);
        const float hn = av[2] + bhn;
        const float n = tanh_hw(pv[2] + r * hn);
        hnew = (1.f - z) * n + z * h_prev;
        h_prev = hnew;
        gv[0] = r; gv[1] = z; gv[G - 1] = n;
        if (a.hn_out) a.hn_out[((size_t)tm * B + bq) * H + j] = hn;
      } else {
        hnew = simple_act<CELL, __nv_bfloat16>(av[0] + pv[0]);
        gv[0] = hnew;
      }
      const size_t bj = (size_t)bq * H + j;
      const unsigned short hb = bf16_bits(hnew);
      hv = hb;
      if (a.gates_out) {
        float* grow = a.gates_out + ((size_t)tm * B + bq) * GH;
#pragma unroll
        for (int g = 0; g < G; ++g) grow[pcol[g]] = gv[g];
      }
      if (CELL == LSTM && a.c_out) a.c_out[(size_t)tm * B * H + bj] = c_state;
      if (a.y) reinterpret_cast<unsigned short*>(a.y)[(size_t)tm * B * H + bj] = hb;
      if (t == a.T - 1) {
        if (a.hT) reinterpret_cast<unsigned short*>(a.hT)[bj] = hb;
        if (CELL == LSTM && a.cT) a.cT[bj] = c_state;
      }
      reinterpret_cast<unsigned short*>(a.hseq)[(size_t)s_out * B * H + bj] = hb;
    }
    // ---- publish
    if constexpr (XCL) {
      // even cell-update threads pair their value with the next unit's and
      // store one tagged word (the warps holding cell-update threads are
      // whole warps here, so the shuffle's mask is every lane)
      if (warp * 32 < uc * B) {
        const uint32_t nbr = __shfl_down_sync(0xffffffffu, hv, 1);
        if (pair && !(q & 1) && !(a.test_skip_publish && blockIdx.x == 0 && t == 0))
          st_relaxed_u64(a.hx + (size_t)(t & 1) * NW + (size_t)blockIdx.x * WS + (q >> 1),
                         ((uint64_t)(t + 1) << 32) | (uint64_t)(hv | (nbr << 16)));
      }
      continue;
    }
    // counter variant: once all of this CTA's h_t stores are done, one
    // release arrival on the step's counter.  When every cell-update thread is
    // in warp 0 a warp barrier orders their stores before lane 0's release.
    if (uc * B <= 32) {
      if (warp == 0) {
        __syncwarp();
        if (lane == 0 && !(a.test_skip_publish && blockIdx.x == 0 && t == 0)) red_release_add(a.arrive + t, 1u);
      }
    } else {
      __syncthreads();
      if (threadIdx.x == 0 && !(a.test_skip_publish && blockIdx.x == 0 && t == 0)) red_release_add(a.arrive + t, 1u);
    }
  }
  // HO = 2: no CTA leaves while a peer may still store into its shared memory
  // (after an abort the peers leave their loops at different steps)
  if constexpr (HO == 2) cluster_barrier();
}

template <int CELL, int MT, int KT, bool W8, int NT>
int launch_one(const Launch& L, const PersistArgs& a, int ctas, bool query_only, int num_sms, int* cl_out) {
  auto kc = persist_fwd_kernel<CELL, MT, KT, 0, W8, NT>;
  auto kx = a.cluster_sync ? persist_fwd_kernel<CELL, MT, KT, 1, W8, NT> : persist_fwd_kernel<CELL, MT, KT, 2, W8, NT>;
  const size_t dyn_w = W8 ? (size_t)MT * 16 * a.H : 0;               // fp8 stash of the CTA's rows
  const size_t dyn = dyn_w + (size_t)2 * a.B * (a.H + 8) * 2;  // + h_{t-1} ping-pong of the cluster variant
  if (dyn_w && cudaFuncSetAttribute(kc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn_w) != cudaSuccess) {
    (void)cudaGetLastError();
    return RNN_ERR_UNSUPPORTED;
  }
  if (query_only) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kc, NT, dyn_w) != cudaSuccess) return RNN_ERR_CUDA;
    if (per_sm * num_sms < ctas) return RNN_ERR_LAUNCH;
    if (cl_out) {
      // the largest cluster size whose clusters all co-reside (0: none)
      *cl_out = 0;
      if (cudaFuncSetAttribute(kx, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn) != cudaSuccess) {
        (void)cudaGetLastError();
        return RNN_OK;
      }
      for (int c = 8; c >= 2; c /= 2) {
        if (ctas % c || (a.H / 2) * a.B / c > NT * kMaxWords) continue;
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3(ctas);
        cfg.blockDim = dim3(NT);
        cfg.dynamicSmemBytes = dyn;
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeClusterDimension;
        at[0].val.clusterDim.x = c;
        at[0].val.clusterDim.y = 1;
        at[0].val.clusterDim.z = 1;
        cfg.attrs = at;
        cfg.numAttrs = 1;
        int nc = 0;
        if (cudaOccupancyMaxActiveClusters(&nc, kx, &cfg) == cudaSuccess && nc * c >= ctas) {
          *cl_out = c;
          break;
        }
        (void)cudaGetLastError();
      }
    }
    return RNN_OK;
  }
  PersistArgs args = a;
  cudaError_t e;
  launch_begin(L);
  if (a.cluster > 0) {
    e = cudaFuncSetAttribute(kx, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn);
    if (e == cudaSuccess) {
      cudaLaunchConfig_t cfg{};
      cfg.gridDim = dim3(ctas);
      cfg.blockDim = dim3(NT);
      cfg.dynamicSmemBytes = dyn;
      cfg.stream = L.stream;
      cudaLaunchAttribute at[2];
      at[0].id = cudaLaunchAttributeClusterDimension;
      at[0].val.clusterDim.x = a.cluster;
      at[0].val.clusterDim.y = 1;
      at[0].val.clusterDim.z = 1;
      at[1].id = cudaLaunchAttributeCooperative;
      at[1].val.cooperative = 1;
      cfg.attrs = at;
      cfg.numAttrs = 2;
      e = cudaLaunchKernelEx(&cfg, kx, args);
    }
  } else {
    void* params[] = {&args};
    e = cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(kc), dim3(ctas), dim3(NT), params, dyn_w, L.stream);
  }
  launch_end(L);
  if (e == cudaErrorCooperativeLaunchTooLarge) return RNN_ERR_LAUNCH;
  return e == cudaSuccess ? RNN_OK : RNN_ERR_CUDA;
}

// (cell, H) -> kernel instance; MT*16 = G*uc rows per CTA, KT*16*8 = H.
// bf16 fragments in registers: LSTM up to H = 1024 (8 units per CTA), GRU up
// to 1024 and the simple RNNs up to 2048 (16 units).  fp8 stash in shared
// memory: LSTM up to 2048 (16 units per CTA from H = 2048, 128 KB of weights),
// GRU up to 2048 (96 KB) and the simple RNNs up to 2048; about 128 CTAs.
int dispatch(const Launch& L, int cell, const PersistArgs& a, bool query_only, int num_sms, int* ctas_out,
             int* cl_out) {
  const int H = a.H;
  const bool w8 = a.Wh8 != nullptr;
  if (H % 128 || a.B < 1 || a.B > 8) return RNN_ERR_UNSUPPORTED;
  int uc = cell == LSTM ? 8 : 16;
  if (w8 && cell == LSTM && H >= 2048) uc = 16;
  const int NT = 256;
  const int KT = H / (16 * (NT / 32));
  const int ctas = H / uc;
  if (ctas_out) *ctas_out = ctas;
  PersistArgs b = a;
  b.uc = uc;
#define RNN_P(C, MT_, KT_) \
  if (cell == C && KT == KT_ && NT == 256) return launch_one<C, MT_, KT_, false, 256>(L, b, ctas, query_only, num_sms, cl_out);
#define RNN_P8(C, MT_, KT_, NT_) \
  if (cell == C && KT == KT_ && NT == NT_ && MT_ * 16 == CellInfo<C>::G * uc) \
    return launch_one<C, MT_, KT_, true, NT_>(L, b, ctas, query_only, num_sms, cl_out);
  if (!w8) {
    RNN_P(LSTM, 2, 1) RNN_P(LSTM, 2, 2) RNN_P(LSTM, 2, 4) RNN_P(LSTM, 2, 8)
    RNN_P(GRU, 3, 1) RNN_P(GRU, 3, 2) RNN_P(GRU, 3, 4) RNN_P(GRU, 3, 8)
    RNN_P(TANH, 1, 1) RNN_P(TANH, 1, 2) RNN_P(TANH, 1, 4) RNN_P(TANH, 1, 8) RNN_P(TANH, 1, 16)
    RNN_P(RELU, 1, 1) RNN_P(RELU, 1, 2) RNN_P(RELU, 1, 4) RNN_P(RELU, 1, 8) RNN_P(RELU, 1, 16)
  } else {
    RNN_P8(LSTM, 2, 1, 256) RNN_P8(LSTM, 2, 2, 256) RNN_P8(LSTM, 2, 4, 256) RNN_P8(LSTM, 2, 8, 256)
    RNN_P8(LSTM, 4, 16, 256)
    RNN_P8(GRU, 3, 1, 256) RNN_P8(GRU, 3, 2, 256) RNN_P8(GRU, 3, 4, 256) RNN_P8(GRU, 3, 8, 256)
    RNN_P8(GRU, 3, 16, 256)
    RNN_P8(TANH, 1, 1, 256) RNN_P8(TANH, 1, 2, 256) RNN_P8(TANH, 1, 4, 256) RNN_P8(TANH, 1, 8, 256)
    RNN_P8(TANH, 1, 16, 256)
    RNN_P8(RELU, 1, 1, 256) RNN_P8(RELU, 1, 2, 256) RNN_P8(RELU, 1, 4, 256) RNN_P8(RELU, 1, 8, 256)
    RNN_P8(RELU, 1, 16, 256)
  }
#undef RNN_P
#undef RNN_P8
  return RNN_ERR_UNSUPPORTED;
}

}  // namespace

int persist_check(int cell, int H, int B, int num_sms, int* ctas, int* cluster, bool fp8) {
  Launch L{};
  PersistArgs a{};
  a.H = H;
  a.B = B;
  static const uint8_t dummy = 0;
  a.Wh8 = fp8 ? &dummy : nullptr;
  return dispatch(L, cell, a, true, num_sms, ctas, cluster);
}

int persist_fwd(const Launch& L, int cell, const PersistArgs& a) {
  int ctas = 0;
  return dispatch(L, cell, a, false, L.num_sms, &ctas, nullptr);
}

}  // namespace rnn
