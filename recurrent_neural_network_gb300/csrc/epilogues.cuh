// epilogues.cuh -- what happens to a finished accumulator tile.
//
//  EpiStore      plain product (+ bias) (+ existing D), float or storage-type
//                output; optional packed->user row remap for weight gradients.
//  EpiFwdStep    the fused recurrent-step update of a forward timestep: the
//                tile holds every gate of u hidden units for 128 batch rows
//                (gate rows are packed in blocks of G*u), so the gate
//                non-linearities and the cell/state update run on the
//                accumulator without it ever reaching memory.
//  EpiBwdStep    the fused backward-through-time step: the accumulator is the
//                recurrent part of dh_{s}; the epilogue adds the gradient
//                arriving from above, runs the pointwise gate derivative of
//                step s and writes the gate gradients that feed the next
//                (earlier) step's product and the weight-gradient GEMMs.
//                Supports split-K with a last-arriving-CTA reduction.
//
// Cell equations (textbook forms of the cells named on the review page of
// "Optimizing Performance of Recurrent Neural Networks on GPUs", section
// "제안 방법"):
//   LSTM: i,f,o = sigmoid, g = tanh; c' = f c + i g; h' = o tanh(c')
//   GRU:  r,z = sigmoid; n = tanh(x_n + r (W_hn h + b_hn)); h' = (1-z) n + z h
//   RNN:  h' = tanh(a)
#pragma once

#include "common.cuh"
#include "engine.cuh"
#include "tc.cuh"

namespace rnn {

// ---------------------------------------------------------------------------
template <class OutT>
struct EpiStore {
  OutT* D;
  long long ldd;
  int M, N;
  const float* bias;  // [N] or null
  int accumulate;     // add to the existing D
  // packed -> user row remap (weight gradients): row p of the product is
  // gate row g of hidden unit j, stored at user row g*H + j.
  int remap, G, u, H;

  __device__ __forceinline__ void prefetch(const TileCoord&, int, int) const {}

  __device__ __forceinline__ long long out_row(int m) const {
    if (!remap) return m;
    const int blk = m / (G * u), r = m % (G * u);
    return (long long)(r / u) * H + (long long)blk * u + (r % u);
  }

  template <class Acc>
  __device__ __forceinline__ void operator()(const TileCoord& t, int row, const Acc& acc, int bn) const {
    const int m = t.m0 + row;
    const bool vec = (N % 16 == 0) && (ldd % 4 == 0);
    for (int c = 0; c < bn; c += 16) {
      float v[16];
      acc.load16(c, v);
      const int n = t.n0 + c;
      if (m >= M || n >= N) continue;
      OutT* dst = D + out_row(m) * ldd + n;
      if (bias) {
#pragma unroll
        for (int i = 0; i < 16; ++i)
          if (n + i < N) v[i] += bias[n + i];
      }
      if (vec && n + 16 <= N) {
        if (accumulate) {
          float o[16];
          load16(dst, o);
#pragma unroll
          for (int i = 0; i < 16; ++i) v[i] += o[i];
        }
        store16(dst, v);
      } else {
        for (int i = 0; i < 16 && n + i < N; ++i) {
          float o = accumulate ? to_f32(dst[i]) : 0.f;
          dst[i] = from_f32<OutT>(v[i] + o);
        }
      }
    }
  }
};

// ---------------------------------------------------------------------------
// Forward step: acc[b][g*u + c] = (h_{t-1} W_h^T)[b][packed(g, j)] for the
// tile's block of u hidden units.
template <int CELL, class S>
struct EpiFwdStep {
  int B, H, u;
  float* P;              // [B][G*H] this step: input projection incl. bias; activated gates written back if write_gates
  int write_gates;
  const float* bias_hn;  // GRU: [H]
  const float* c_prev;   // LSTM [B][H], null = zero
  float* c_out;          // LSTM [B][H]
  const S* h_prev;       // [B][H] (GRU), null = zero
  S* h_out;              // [B][H]
  S* y;                  // [B][H] or null
  S* hT;                 // [B][H] or null
  float* cT;             // [B][H] or null
  float* hn_out;         // GRU [B][H] or null

  __device__ __forceinline__ void prefetch(const TileCoord& t, int row, int /*bn*/) const {
    constexpr int G = CellInfo<CELL>::G;
    const int b = t.m0 + row;
    if (b >= B) return;
    const int jblk = (t.n0 / (G * u)) * u;
    tc::prefetch_l2(P + (size_t)b * G * H + t.n0, G * u * 4);
    if (CELL == LSTM && c_prev) tc::prefetch_l2(c_prev + (size_t)b * H + jblk, u * 4);
    if (CELL == GRU && h_prev) tc::prefetch_l2(h_prev + (size_t)b * H + jblk, u * sizeof(S));
  }

  template <class Acc>
  __device__ __forceinline__ void operator()(const TileCoord& t, int row, const Acc& acc, int /*bn*/) const {
    constexpr int G = CellInfo<CELL>::G;
    const int b = t.m0 + row;
    const int GH = G * H;
    const int jblk = (t.n0 / (G * u)) * u;
    for (int c = 0; c < u; c += 16) {
      float a[G][16];
#pragma unroll
      for (int g = 0; g < G; ++g) acc.load16(g * u + c, a[g]);
      if (b >= B) continue;
      const int j0 = jblk + c;
      float* prow = P + (size_t)b * GH + t.n0 + c;
      float hnew[16];
      if constexpr (CELL == LSTM) {
        float cp[16];
        if (c_prev) load16(c_prev + (size_t)b * H + j0, cp);
        else
#pragma unroll
          for (int i = 0; i < 16; ++i) cp[i] = 0.f;
        float p[16], cn[16];
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          load16(prow + g * u, p);
#pragma unroll
          for (int i = 0; i < 16; ++i) a[g][i] += p[i];
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float ig = Act<S>::sig(a[0][i]), fg = Act<S>::sig(a[1][i]), gg = Act<S>::th(a[2][i]), og = Act<S>::sig(a[3][i]);
          const float cc = fg * cp[i] + ig * gg;
          cn[i] = cc;
          hnew[i] = og * Act<S>::th(cc);
          a[0][i] = ig; a[1][i] = fg; a[2][i] = gg; a[3][i] = og;
        }
        store16(c_out + (size_t)b * H + j0, cn);
        if (cT) store16(cT + (size_t)b * H + j0, cn);
      } else if constexpr (CELL == GRU) {
        float hp[16], p[16], bn[16], hn[16];
        if (h_prev) load16(h_prev + (size_t)b * H + j0, hp);
        else
#pragma unroll
          for (int i = 0; i < 16; ++i) hp[i] = 0.f;
        load16(bias_hn + j0, bn);
#pragma unroll
        for (int g = 0; g < 2; ++g) {
          load16(prow + g * u, p);
#pragma unroll
          for (int i = 0; i < 16; ++i) a[g][i] += p[i];
        }
        load16(prow + 2 * u, p);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float r = Act<S>::sig(a[0][i]), z = Act<S>::sig(a[1][i]);
          hn[i] = a[2][i] + bn[i];
          const float n = Act<S>::th(p[i] + r * hn[i]);
          hnew[i] = (1.f - z) * n + z * hp[i];
          a[0][i] = r; a[1][i] = z; a[2][i] = n;
        }
        if (hn_out) store16(hn_out + (size_t)b * H + j0, hn);
      } else {
        float p[16];
        load16(prow, p);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          hnew[i] = Act<S>::th(a[0][i] + p[i]);
          a[0][i] = hnew[i];
        }
      }
      if (write_gates) {
#pragma unroll
        for (int g = 0; g < G; ++g) store16(prow + g * u, a[g]);
      }
      store16(h_out + (size_t)b * H + j0, hnew);
      if (y) store16(y + (size_t)b * H + j0, hnew);
      if (hT) store16(hT + (size_t)b * H + j0, hnew);
    }
  }
};

// ---------------------------------------------------------------------------
// Backward pointwise of step s for 16 hidden units j0..j0+15 of batch row b.
// dh: recurrent gradient reaching h_s (without the gradient from above and
// without the GRU direct term; both are added here).
template <int CELL, class S>
struct BwdPoint {
  int B, H, u;
  const float* gates;   // [B][G*H] activated gates of step s
  const float* c_s;     // LSTM [B][H]
  const float* c_sm1;   // LSTM [B][H] (c_{s-1}, c0 for s = 0), null = zero
  const float* hn_s;    // GRU [B][H]
  const S* h_sm1;       // GRU [B][H] (h_{s-1}), null = zero
  const void* dy;       // [B][H] gradient from above at step s (float if dy_f32 else S)
  int dy_f32;
  float* carry;         // LSTM: dc flowing into step s (in) / into s-1 (out). GRU: dh_{s+1} z_{s+1} (in) / dh_s z_s (out)
  S* dGx;               // [B][G*H]
  S* dGh;               // [B][G*H] (GRU; LSTM/RNN write only dGx)

  __device__ __forceinline__ void run(int b, int j0, float* dh) const {
    constexpr int G = CellInfo<CELL>::G;
    const int GH = G * H;
    const size_t bj = (size_t)b * H + j0;
    float t16[16];
    if (dy) {
      if (dy_f32) load16(reinterpret_cast<const float*>(dy) + bj, t16);
      else load16(reinterpret_cast<const S*>(dy) + bj, t16);
#pragma unroll
      for (int i = 0; i < 16; ++i) dh[i] += t16[i];
    }
    const int p0 = (j0 / u) * (G * u) + (j0 % u);  // packed column of gate 0
    const float* grow = gates + (size_t)b * GH + p0;
    S* gx = dGx + (size_t)b * GH + p0;
    if constexpr (CELL == LSTM) {
      float ig[16], fg[16], gg[16], og[16], cs[16], cp[16], dc[16];
      load16(grow, ig);
      load16(grow + u, fg);
      load16(grow + 2 * u, gg);
      load16(grow + 3 * u, og);
      load16(c_s + bj, cs);
      if (c_sm1) load16(c_sm1 + bj, cp);
      else
#pragma unroll
        for (int i = 0; i < 16; ++i) cp[i] = 0.f;
      load16(carry + bj, dc);
      float d0[16], d1[16], d2[16], d3[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float tau = Act<S>::th(cs[i]);
        const float dov = dh[i] * tau;
        const float dcv = dc[i] + dh[i] * og[i] * (1.f - tau * tau);
        d0[i] = dcv * gg[i] * ig[i] * (1.f - ig[i]);
        d1[i] = dcv * cp[i] * fg[i] * (1.f - fg[i]);
        d2[i] = dcv * ig[i] * (1.f - gg[i] * gg[i]);
        d3[i] = dov * og[i] * (1.f - og[i]);
        dc[i] = dcv * fg[i];
      }
      store16(gx, d0);
      store16(gx + u, d1);
      store16(gx + 2 * u, d2);
      store16(gx + 3 * u, d3);
      store16(carry + bj, dc);
    } else if constexpr (CELL == GRU) {
      float r[16], z[16], n[16], hn[16], hp[16], cz[16];
      load16(grow, r);
      load16(grow + u, z);
      load16(grow + 2 * u, n);
      load16(hn_s + bj, hn);
      if (h_sm1) load16(h_sm1 + bj, hp);
      else
#pragma unroll
        for (int i = 0; i < 16; ++i) hp[i] = 0.f;
      load16(carry + bj, cz);
      float dar[16], daz[16], dan[16], dhn[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float d = dh[i] + cz[i];
        const float dn = d * (1.f - z[i]);
        const float dz = d * (hp[i] - n[i]);
        dan[i] = dn * (1.f - n[i] * n[i]);
        const float dr = dan[i] * hn[i];
        dhn[i] = dan[i] * r[i];
        dar[i] = dr * r[i] * (1.f - r[i]);
        daz[i] = dz * z[i] * (1.f - z[i]);
        cz[i] = d * z[i];
      }
      S* gh = dGh + (size_t)b * GH + p0;
      store16(gx, dar);
      store16(gx + u, daz);
      store16(gx + 2 * u, dan);
      store16(gh, dar);
      store16(gh + u, daz);
      store16(gh + 2 * u, dhn);
      store16(carry + bj, cz);
    } else {
      float hv[16], da[16];
      load16(grow, hv);
#pragma unroll
      for (int i = 0; i < 16; ++i) da[i] = dh[i] * (1.f - hv[i] * hv[i]);
      store16(gx, da);
    }
  }
};

// ---------------------------------------------------------------------------
// Backward step.  The product is acc[b][j] = (dGh_{s+1} W_h)[b][j] over a
// tile of hidden units j; `final` (s = -1) writes dh0 / dc0 instead of
// running a pointwise step.
template <int CELL, class S>
struct EpiBwdStep {
  BwdPoint<CELL, S> pt;
  int final_;
  S* dh0;        // [B][H] (final)
  float* dc0;    // [B][H] (final, LSTM)
  float* part;   // split-K partials [splits][B][H] (global-memory reduction)
  int* counters; // one per (m-tile, n-tile), zero before the first use
  int* err;      // device error word (cluster reduction waits)
  uint64_t limit_ns;

  __device__ __forceinline__ void finish(int b, int j0, float* dh) const {
    const int H = pt.H;
    if (!final_) {
      pt.run(b, j0, dh);
      return;
    }
    const size_t bj = (size_t)b * H + j0;
    if (CELL == GRU) {
      float cz[16];
      load16(pt.carry + bj, cz);
#pragma unroll
      for (int i = 0; i < 16; ++i) dh[i] += cz[i];
    }
    if (dh0) store16(dh0 + bj, dh);
    if (CELL == LSTM && dc0) {
      float dc[16];
      load16(pt.carry + bj, dc);
      store16(dc0 + bj, dc);
    }
  }

  // Rows are shared out over the split-K CTAs of the tile: whichever of them
  // arrives last finds its inputs in L2.
  __device__ __forceinline__ void prefetch(const TileCoord& t, int row, int bn) const {
    constexpr int G = CellInfo<CELL>::G;
    const int b = t.m0 + row;
    const int B = pt.B, H = pt.H;
    if (b >= B || final_ || (row % t.splits) != t.split) return;
    const int nu = min(bn, H - t.n0);  // units of this tile (a multiple of u)
    const size_t bj = (size_t)b * H + t.n0;
    const int p0 = (t.n0 / pt.u) * (G * pt.u);
    tc::prefetch_l2(pt.gates + (size_t)b * G * H + p0, nu * G * 4);
    if (CELL == LSTM) {
      tc::prefetch_l2(pt.c_s + bj, nu * 4);
      if (pt.c_sm1) tc::prefetch_l2(pt.c_sm1 + bj, nu * 4);
    }
    if (CELL == GRU) {
      tc::prefetch_l2(pt.hn_s + bj, nu * 4);
      if (pt.h_sm1) tc::prefetch_l2(pt.h_sm1 + bj, nu * sizeof(S));
    }
    if (CELL != TANH) tc::prefetch_l2(pt.carry + bj, nu * 4);
    if (pt.dy) tc::prefetch_l2(static_cast<const char*>(pt.dy) + bj * (pt.dy_f32 ? 4 : sizeof(S)),
                               nu * (pt.dy_f32 ? 4 : (int)sizeof(S)));
  }

  template <class Acc>
  __device__ __forceinline__ void operator()(const TileCoord& t, int row, const Acc& acc, int bn) const {
    const int b = t.m0 + row;
    const int B = pt.B, H = pt.H;
    if (t.splits > 1 && t.cluster > 1) {
      // Split-K partials reduced across the cluster: every CTA parks its
      // partial tile in its own shared memory, then CTA `split` sums columns
      // [split*cw, (split+1)*cw) over all CTAs through distributed shared
      // memory and runs the pointwise step for those hidden units.
      const int RS = bn + 4;
      const int lane = threadIdx.x & 31;
      float* mine = t.red + (size_t)row * RS;
      for (int c = 0; c < bn; c += 16) {
        float v[16];
        acc.load16(c, v);
        float4* d = reinterpret_cast<float4*>(mine + c);
#pragma unroll
        for (int q = 0; q < 4; ++q) d[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
      }
      tc::fence_acq_rel_cluster();
      __syncwarp();
      const uint32_t full_local = tc::smem_addr(t.red_full), done_local = tc::smem_addr(t.red_done);
      if (lane == 0)
        for (int p = 0; p < t.cluster; ++p) tc::mbar_arrive_remote(tc::mapa(full_local, t.peer_base + p * t.peer_stride));
      int ok = 1;
      if (lane == 0) ok = tc::mbar_wait_cluster(t.red_full, 0, err, limit_ns) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (ok && b < B) {
        const int cw = bn / t.cluster;
        const uint32_t mine_addr = tc::smem_addr(mine);
        for (int c = t.split * cw; c < (t.split + 1) * cw; c += 16) {
          const int j0 = t.n0 + c;
          if (j0 >= H) break;
          float v[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) v[i] = 0.f;
          for (int p = 0; p < t.cluster; ++p) {
            const uint32_t ra = tc::mapa(mine_addr, t.peer_base + p * t.peer_stride) + c * 4;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              float w[4];
              tc::ld_dsmem4(ra + 16 * q, w);
              v[4 * q] += w[0]; v[4 * q + 1] += w[1]; v[4 * q + 2] += w[2]; v[4 * q + 3] += w[3];
            }
          }
          finish(b, j0, v);
        }
      }
      tc::fence_acq_rel_cluster();
      __syncwarp();
      if (lane == 0)
        for (int p = 0; p < t.cluster; ++p) tc::mbar_arrive_remote(tc::mapa(done_local, t.peer_base + p * t.peer_stride));
      if (lane == 0) tc::mbar_wait_cluster(t.red_done, 0, err, limit_ns);
      __syncwarp();
      return;
    }
    if (t.splits > 1) {
      // write this split's partial, then the last CTA of the tile reduces
      for (int c = 0; c < bn; c += 16) {
        float v[16];
        acc.load16(c, v);
        if (b < B && t.n0 + c < H) store16(part + ((size_t)t.split * B + b) * H + t.n0 + c, v);
      }
      __threadfence();
      asm volatile("bar.sync 1, 128;" ::: "memory");
      if (row == 0) {
        int* ctr = counters + t.mt * ((H + bn - 1) / bn) + t.nt;
        const int old = atomicAdd(ctr, 1);
        const int last = (old == t.splits - 1);
        if (last) *ctr = 0;
        t.scratch[0] = last;
      }
      asm volatile("bar.sync 1, 128;" ::: "memory");
      const int last = *reinterpret_cast<volatile int*>(t.scratch);
      if (!last) return;
      __threadfence();
      if (b >= B) return;
      for (int c = 0; c < bn; c += 16) {
        const int j0 = t.n0 + c;
        if (j0 >= H) break;
        float v[16], o[16];
        load16_cg(part + ((size_t)t.split * B + b) * H + j0, v);
        for (int sp = 0; sp < t.splits; ++sp) {
          if (sp == t.split) continue;
          load16_cg(part + ((size_t)sp * B + b) * H + j0, o);
#pragma unroll
          for (int i = 0; i < 16; ++i) v[i] += o[i];
        }
        finish(b, j0, v);
      }
      return;
    }
    for (int c = 0; c < bn; c += 16) {
      float v[16];
      acc.load16(c, v);
      const int j0 = t.n0 + c;
      if (b < B && j0 < H) finish(b, j0, v);
    }
  }
};

}  // namespace rnn
