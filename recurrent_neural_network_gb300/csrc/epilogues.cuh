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
  // fp32 storage (the FFMA engine): the pointwise work, in double precision,
  // is shared out over at least four threads per tile row, each taking every
  // fourth element of a 16-unit chunk (TileCoord::part of TileCoord::parts;
  // more shares where the tile has few rows)
  static constexpr int kSimtShares = std::is_same<S, float>::value ? 4 : 1;
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
    using T = typename Prec<S>::T;  // pointwise precision
    const int b = t.m0 + row;
    const int GH = G * H;
    const int jblk = (t.n0 / (G * u)) * u;
    // this thread's share: every es-th element of a chunk from e; beyond 16
    // shares the chunks are shared out too (cs threads per element)
    const int sh = kSimtShares == 1 ? 1 : t.parts, s = kSimtShares == 1 ? 0 : t.part;
    const int es = sh > 16 ? 16 : sh, e = s & (es - 1), cs = sh / es, c0 = (s / es) * 16;
    for (int c = c0; c < u; c += 16 * cs) {
      float a[G][16];
#pragma unroll
      for (int g = 0; g < G; ++g) acc.load16(g * u + c, a[g]);
      if (b >= B) continue;
      const int j0 = jblk + c;
      float* prow = P + (size_t)b * GH + t.n0 + c;
      float hnew[16] = {};
      if constexpr (CELL == LSTM) {
        float cp[16];
        if (c_prev) load16(c_prev + (size_t)b * H + j0, cp);
        else
#pragma unroll
          for (int i = 0; i < 16; ++i) cp[i] = 0.f;
        float p[16], cn[16] = {};
        T av[4][16];
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          load16(prow + g * u, p);
#pragma unroll
          for (int i = 0; i < 16; ++i) av[g][i] = T(a[g][i]) + T(p[i]);
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          if ((i & (es - 1)) != e) continue;
          const T ig = Act<S>::sig(av[0][i]), fg = Act<S>::sig(av[1][i]), gg = Act<S>::th(av[2][i]),
                  og = Act<S>::sig(av[3][i]);
          const T cc = fg * T(cp[i]) + ig * gg;
          cn[i] = float(cc);
          hnew[i] = float(og * Act<S>::th(cc));
          a[0][i] = float(ig); a[1][i] = float(fg); a[2][i] = float(gg); a[3][i] = float(og);
        }
        store16_share(c_out + (size_t)b * H + j0, cn, e, es);
        if (cT) store16_share(cT + (size_t)b * H + j0, cn, e, es);
      } else if constexpr (CELL == GRU) {
        float hp[16], p[16], bn[16], hn[16] = {};
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
          if ((i & (es - 1)) != e) continue;
          const T r = Act<S>::sig(T(a[0][i])), z = Act<S>::sig(T(a[1][i]));
          const T hnv = T(a[2][i]) + T(bn[i]);
          hn[i] = float(hnv);
          const T n = Act<S>::th(T(p[i]) + r * hnv);
          hnew[i] = float((T(1) - z) * n + z * T(hp[i]));
          a[0][i] = float(r); a[1][i] = float(z); a[2][i] = float(n);
        }
        if (hn_out) store16_share(hn_out + (size_t)b * H + j0, hn, e, es);
      } else {
        float p[16];
        load16(prow, p);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          if ((i & (es - 1)) != e) continue;
          hnew[i] = float(simple_act<CELL, S>(T(a[0][i]) + T(p[i])));
          a[0][i] = hnew[i];
        }
      }
      if (write_gates) {
#pragma unroll
        for (int g = 0; g < G; ++g) store16_share(prow + g * u, a[g], e, es);
      }
      store16_share(h_out + (size_t)b * H + j0, hnew, e, es);
      if (y) store16_share(y + (size_t)b * H + j0, hnew, e, es);
      if (hT) store16_share(hT + (size_t)b * H + j0, hnew, e, es);
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

  // e, es: this thread's share of the 16 elements (every es-th from e; es a
  // power of two), as the forward step's FFMA epilogue shares them out
  __device__ __forceinline__ void run(int b, int j0, float* dh32, int e = 0, int es = 1) const {
    constexpr int G = CellInfo<CELL>::G;
    using T = typename Prec<S>::T;  // pointwise precision
    const int GH = G * H;
    const size_t bj = (size_t)b * H + j0;
    T dh[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) dh[i] = T(dh32[i]);
    float t16[16];
    if (dy) {
      if (dy_f32) load16(reinterpret_cast<const float*>(dy) + bj, t16);
      else load16(reinterpret_cast<const S*>(dy) + bj, t16);
#pragma unroll
      for (int i = 0; i < 16; ++i) dh[i] += T(t16[i]);
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
      float d0[16] = {}, d1[16] = {}, d2[16] = {}, d3[16] = {};
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        if ((i & (es - 1)) != e) continue;
        const T igv = ig[i], fgv = fg[i], ggv = gg[i], ogv = og[i];
        const T tau = Act<S>::th(T(cs[i]));
        const T dov = dh[i] * tau;
        const T dcv = T(dc[i]) + dh[i] * ogv * (T(1) - tau * tau);
        d0[i] = float(dcv * ggv * igv * (T(1) - igv));
        d1[i] = float(dcv * T(cp[i]) * fgv * (T(1) - fgv));
        d2[i] = float(dcv * igv * (T(1) - ggv * ggv));
        d3[i] = float(dov * ogv * (T(1) - ogv));
        dc[i] = float(dcv * fgv);
      }
      store16_share(gx, d0, e, es);
      store16_share(gx + u, d1, e, es);
      store16_share(gx + 2 * u, d2, e, es);
      store16_share(gx + 3 * u, d3, e, es);
      store16_share(carry + bj, dc, e, es);
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
      float dar[16] = {}, daz[16] = {}, dan[16] = {}, dhn[16] = {};
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        if ((i & (es - 1)) != e) continue;
        const T rv = r[i], zv = z[i], nv = n[i];
        const T d = dh[i] + T(cz[i]);
        const T dn = d * (T(1) - zv);
        const T dz = d * (T(hp[i]) - nv);
        const T danv = dn * (T(1) - nv * nv);
        const T dr = danv * T(hn[i]);
        dan[i] = float(danv);
        dhn[i] = float(danv * rv);
        dar[i] = float(dr * rv * (T(1) - rv));
        daz[i] = float(dz * zv * (T(1) - zv));
        cz[i] = float(d * zv);
      }
      S* gh = dGh + (size_t)b * GH + p0;
      store16_share(gx, dar, e, es);
      store16_share(gx + u, daz, e, es);
      store16_share(gx + 2 * u, dan, e, es);
      store16_share(gh, dar, e, es);
      store16_share(gh + u, daz, e, es);
      store16_share(gh + 2 * u, dhn, e, es);
      store16_share(carry + bj, cz, e, es);
    } else {
      float hv[16], da[16] = {};
      load16(grow, hv);
#pragma unroll
      for (int i = 0; i < 16; ++i)
        if ((i & (es - 1)) == e) da[i] = float(dh[i] * simple_slope<CELL>(T(hv[i])));
      store16_share(gx, da, e, es);
    }
  }
};

// ---------------------------------------------------------------------------
// Backward step.  The product is acc[b][j] = (dGh_{s+1} W_h)[b][j] over a
// tile of hidden units j; `final` (s = -1) writes dh0 / dc0 instead of
// running a pointwise step.
template <int CELL, class S>
struct EpiBwdStep {
  // fp32 storage (the FFMA engine): at least four threads per tile row share
  // out the double-precision pointwise work (more where the tile has few rows)
  static constexpr int kSimtShares = std::is_same<S, float>::value ? 4 : 1;
  BwdPoint<CELL, S> pt;
  int final_;
  S* dh0;        // [B][H] (final)
  float* dc0;    // [B][H] (final, LSTM)
  float* part;   // split-K partials [splits][B][H] (global-memory reduction)
  int* counters; // one per (m-tile, n-tile), zero before the first use
  int* err;      // device error word (cluster reduction waits)
  uint64_t limit_ns;

  __device__ __forceinline__ void finish(int b, int j0, float* dh, int e = 0, int es = 1) const {
    const int H = pt.H;
    if (!final_) {
      pt.run(b, j0, dh, e, es);
      return;
    }
    const size_t bj = (size_t)b * H + j0;
    if (CELL == GRU) {
      float cz[16];
      load16(pt.carry + bj, cz);
#pragma unroll
      for (int i = 0; i < 16; ++i) dh[i] += cz[i];
    }
    if (dh0) store16_share(dh0 + bj, dh, e, es);
    if (CELL == LSTM && dc0) {
      float dc[16];
      load16(pt.carry + bj, dc);
      store16_share(dc0 + bj, dc, e, es);
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
    if (CELL == LSTM || CELL == GRU) tc::prefetch_l2(pt.carry + bj, nu * 4);
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
    // (the FFMA engine's shares of a row; one share in the tensor-core engines)
    const int sh = kSimtShares == 1 ? 1 : t.parts, s = kSimtShares == 1 ? 0 : t.part;
    const int es = sh > 16 ? 16 : sh, e = s & (es - 1), cs = sh / es, c0 = (s / es) * 16;
    for (int c = c0; c < bn; c += 16 * cs) {
      float v[16];
      acc.load16(c, v);
      const int j0 = t.n0 + c;
      if (b < B && j0 < H) finish(b, j0, v, e, es);
    }
  }
};

// ---------------------------------------------------------------------------
// Transposed recurrent steps.  With many gate rows and at most a few hundred
// batch rows the step product is taken as W_h h^T instead of h W_h^T: tile
// rows are packed gate rows (forward) or hidden units (backward) and tile
// columns are batch entries.  A warp's 32 TMEM lanes are then 32 consecutive
// rows, so each of its global accesses in the epilogue is one contiguous run
// (the batch-row-per-thread layout above touches 32 separate lines per
// access).  These epilogues use the packing unit u = 1: packed row G*j + g is
// gate g of hidden unit j, so the four LSTM gates of a unit sit in four
// neighbouring lanes of one warp.

// a[s] for a lane-dependent s in 0..3 without local-memory indexing
__device__ __forceinline__ float pick4(float a0, float a1, float a2, float a3, int s) {
  const float lo = (s & 1) ? a1 : a0, hi = (s & 1) ? a3 : a2;
  return (s & 2) ? hi : lo;
}

// Forward step, tile = 128 packed gate rows (one CTA of a pair) x bn batch
// entries.  acc[p][b] = (W_h h_{t-1}^T)[p][b].  When the CTA owns a single
// tile, stage() moves this tile's slice of P into the idle second TMEM
// accumulator (and the LSTM c_{t-1} values into registers) while the MMAs
// run, so the epilogue proper only reads TMEM and stores.
template <int CELL>
struct EpiFwdStepT {
  static constexpr int kWarps = 8;  // two warps per TMEM lane quadrant, each half of the columns
  using S = __nv_bfloat16;
  static constexpr int kAhead = 4;  // chunks of c_{t-1} loaded ahead of their use
  struct Stash {
    float cp[kAhead][4];  // LSTM c_{t-1} of the next kAhead chunks
  };
  static constexpr int kUnits = 128 / CellInfo<CELL>::G;  // hidden units of a 128-row tile
  // Bulk-store maps of the single-tile path (tma_out): the epilogue writes
  // gates, c and h as [batch][row] tiles into its idle pipeline buffers and
  // stores every 32 finished batch rows with bulk tensor copies (boxes of 128
  // gate rows or kUnits units x 32 batch entries) while it computes the next.
  CUtensorMap map_p, map_c, map_h, map_y, map_hT, map_cT;
  int tma_out;
  int B, H;
  float* P;          // [B][G*H] this step: input projection incl. bias; activated gates written back if write_gates
  int write_gates;
  const float* c_prev;  // LSTM [B][H], null = zero
  float* c_out;         // LSTM [B][H]
  S* h_out;             // [B][H]
  S* y;                 // [B][H] or null
  S* hT;                // [B][H] or null
  float* cT;            // [B][H] or null
  // launches over several dependent steps (TileCoord::step): P, c, h and y
  // are the chunk's sequences, step s at rows step_rows * s further (c_prev
  // the row block before c_out's: step s reads step s-1's c); hT / cT are
  // written by step hT_step only; after its stores of step s are complete
  // each storing thread arrives on step_cnt[s]
  int step_rows, hT_step;
  unsigned int* step_cnt;

  __device__ __forceinline__ void prefetch(const TileCoord& t, int row, int bn) const {
    constexpr int G = CellInfo<CELL>::G;
    const int GH = G * H;
    if (t.m0 >= GH) return;
    const int rows = min(128, GH - t.m0);
    for (int i = row; i < bn; i += 128) {
      const int b = t.n0 + i + t.step * step_rows;
      if (b >= B) break;
      tc::prefetch_l2(P + (size_t)b * GH + t.m0, rows * 4);
      if (CELL == LSTM && c_prev) tc::prefetch_l2(c_prev + (size_t)b * H + t.m0 / 4, rows);
    }
  }

  // c_{t-1} for the (unit p/4, batch entry c + 4k + p%4) pairs of chunk c;
  // in the cell update from the shared-memory gate tile (smem_map) a lane
  // takes instead unit (first unit of its warp) + lane % 8, batch entry
  // c + 4k + lane / 8
  __device__ __forceinline__ void load_cp(int n0, int p, bool live, int c, int nmax, float* cp,
                                          bool smem_map = false) const {
    int g = p & 3, j = p >> 2;
    if (smem_map) {
      const int lane = threadIdx.x & 31;
      g = lane >> 3;
      j = ((p & ~31) >> 2) + (lane & 7);
      live = j < H;
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int bi = c + 4 * k + g;
      cp[k] = (live && c_prev && bi < nmax) ? c_prev[(size_t)(n0 + bi) * H + j] : 0.f;
    }
  }

  // v: pre-activations (P included) of gate row p for batch entries c..c+15.
  // With sm_g non-null the outputs go to the shared-memory tiles sm_g
  // ([bn][128] gates), sm_c / sm_h ([bn][kUnits]) at tile row `row`.
  __device__ __forceinline__ void finish(int n0, int p, bool live, int c, int nb, float* v, const float* cp,
                                         int row = 0, float* sm_g = nullptr, float* sm_c = nullptr,
                                         S* sm_h = nullptr) const {
    constexpr int G = CellInfo<CELL>::G;
    const int GH = G * H;
    float* pc = P + (size_t)(n0 + c) * GH + p;
    if constexpr (CELL == LSTM) {
      // g = p % 4: input, forget, cell candidate (tanh), output gate
      const int g = p & 3;
      const float sc = g == 2 ? 1.f : 0.5f;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float th = tanh_hw(sc * v[i]);
        v[i] = g == 2 ? th : fmaf(0.5f, th, 0.5f);
      }
      if (sm_g) {
#pragma unroll
        for (int i = 0; i < 16; ++i) sm_g[(c + i) * 128 + row] = v[i];
        // the warp's 32 gate rows (8 units) of these 16 batch entries are in
        // the tile: lane (u, e) = (lane & 7, lane >> 3) reads the four gates of
        // unit u for batch entry c + 4k + e as one 16-byte vector (each 8-lane
        // phase reads 128 contiguous bytes)
        __syncwarp();
        const int lane = threadIdx.x & 31, rw = row & ~31;
        const int ul = rw / 4 + (lane & 7), e = lane >> 3;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int bi = 4 * k + e;
          const float4 gt = *reinterpret_cast<const float4*>(sm_g + (c + bi) * 128 + rw + 4 * (lane & 7));
          const float cn = gt.y * cp[k] + gt.x * gt.z;
          const float hn = gt.w * tanh_hw(cn);
          sm_c[(c + bi) * kUnits + ul] = cn;
          sm_h[(c + bi) * kUnits + ul] = __float2bfloat16_rn(hn);
        }
        return;
      }
      if (write_gates && live) {
#pragma unroll
        for (int i = 0; i < 16; ++i)
          if (i < nb) pc[(size_t)i * GH] = v[i];
      }
      // 4 x 4 transposes within each group of four lanes: afterwards lane g
      // of unit j holds all four gates of j for batch entry c + 4k + g
      const int j = p >> 2;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float q0 = v[4 * k], q1 = v[4 * k + 1], q2 = v[4 * k + 2], q3 = v[4 * k + 3];
        float gt[4];
        gt[0] = gt[1] = gt[2] = gt[3] = pick4(q0, q1, q2, q3, g);
#pragma unroll
        for (int r = 1; r < 4; ++r) {
          const float got = __shfl_xor_sync(0xffffffffu, pick4(q0, q1, q2, q3, g ^ r), r);
          const int src = g ^ r;  // the lane holding gate src sent its value for batch entry c + 4k + g
          gt[0] = src == 0 ? got : gt[0];
          gt[1] = src == 1 ? got : gt[1];
          gt[2] = src == 2 ? got : gt[2];
          gt[3] = src == 3 ? got : gt[3];
        }
        const int bi = 4 * k + g;
        const float cn = gt[1] * cp[k] + gt[0] * gt[2];
        const float hn = gt[3] * tanh_hw(cn);
        const S hb = __float2bfloat16_rn(hn);
        if (!live || bi >= nb) continue;
        const size_t bj = (size_t)(n0 + c + bi) * H + j;
        c_out[bj] = cn;
        if (cT) cT[bj] = cn;
        h_out[bj] = hb;
        if (y) y[bj] = hb;
        if (hT) hT[bj] = hb;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) v[i] = simple_act<CELL, S>(v[i]);
      if (sm_g) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          sm_g[(c + i) * 128 + row] = v[i];
          sm_h[(c + i) * kUnits + row] = __float2bfloat16_rn(v[i]);
        }
      } else if (live) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          if (i >= nb) continue;
          if (write_gates) pc[(size_t)i * GH] = v[i];
          const size_t bj = (size_t)(n0 + c + i) * H + p;
          const S hb = __float2bfloat16_rn(v[i]);
          h_out[bj] = hb;
          if (y) y[bj] = hb;
          if (hT) hT[bj] = hb;
        }
      }
    }
  }

  template <class Acc>
  __device__ __forceinline__ void operator()(const TileCoord& t, int row, const Acc& acc, int bn) const {
    constexpr int G = CellInfo<CELL>::G;
    const int GH = G * H;
    const int p = t.m0 + row;  // packed gate row of this lane
    const bool live = p < GH;
    const int cw = bn / t.parts, cb = t.part * cw;
    const int nmax = min(cb + cw, B - t.n0);
#pragma unroll 1
    for (int c = cb; c < nmax; c += 16) {
      float v[16], pv[16], cp[4];
      const int nb = min(16, nmax - c);
      const int rn = t.n0 + t.step * step_rows;
      const float* pc = P + (size_t)(rn + c) * GH + p;
#pragma unroll
      for (int i = 0; i < 16; ++i) pv[i] = (live && i < nb) ? pc[(size_t)i * GH] : 0.f;
      if (CELL == LSTM) load_cp(rn, p, live, c, nmax, cp);
      acc.load16(c, v);
#pragma unroll
      for (int i = 0; i < 16; ++i) v[i] += pv[i];
      finish(rn, p, live, c, nb, v, cp);
    }
  }

  __device__ __forceinline__ void stage(const TileCoord& t, int row, uint32_t taddr, int bn, Stash& st) const {
    constexpr int G = CellInfo<CELL>::G;
    const int GH = G * H;
    const int p = t.m0 + row;
    const bool live = p < GH;
    const int cw = bn / t.parts, cb = t.part * cw;
    const int nmax = min(cb + cw, B - t.n0);
    if constexpr (CELL == LSTM) {
#pragma unroll
      for (int a = 0; a < kAhead; ++a)
        load_cp(t.n0 + t.step * step_rows, p, live, cb + 16 * a, nmax, st.cp[a], tma_out);
    }
    // P, two chunks (32 loads per lane) in flight at a time
#pragma unroll 1
    for (int c = cb; c < nmax; c += 32) {
      float v0[16], v1[16];
      const float* pc = P + (size_t)(t.n0 + t.step * step_rows + c) * GH + p;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        v0[i] = (live && c + i < nmax) ? pc[(size_t)i * GH] : 0.f;
        v1[i] = (live && c + 16 + i < nmax) ? pc[(size_t)(16 + i) * GH] : 0.f;
      }
      tc::tmem_store16(taddr + c, v0);
      if (c + 16 < nmax) tc::tmem_store16(taddr + c + 16, v1);
    }
    tc::tmem_store_wait();
  }

  template <class Acc>
  __device__ __forceinline__ void run_staged(const TileCoord& t, int row, const Acc& acc, const Acc& staged, int bn,
                                             Stash& st) const {
    constexpr int G = CellInfo<CELL>::G;
    const int p = t.m0 + row;
    const bool live = p < G * H;
    const int cw = bn / t.parts, cb = t.part * cw;
    const int nmax = min(cb + cw, B - t.n0);
    // output tiles in the pipeline buffers (free once the tile's MMAs are done)
    float* sm_g = t.red;
    float* sm_c = sm_g + (size_t)bn * 128;
    S* sm_h = reinterpret_cast<S*>(sm_c + (CELL == LSTM ? (size_t)bn * kUnits : 0));
    // 32 columns (two chunks) per TMEM round trip; each part is a multiple of 32 wide
#pragma unroll 1
    for (int c2 = cb; c2 < nmax; c2 += 32) {
      float v2[32], pv2[32];
      acc.load32_with(staged, c2, v2, pv2);
#pragma unroll
      for (int i = 0; i < 32; ++i) v2[i] += pv2[i];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int c = c2 + 16 * h;
        if (c >= nmax) break;
        float cp[4];
        if constexpr (CELL == LSTM) {
          // rotate the look-ahead ring and start the loads of chunk c + kAhead
#pragma unroll
          for (int k = 0; k < 4; ++k) cp[k] = st.cp[0][k];
#pragma unroll
          for (int a = 0; a + 1 < kAhead; ++a)
#pragma unroll
            for (int k = 0; k < 4; ++k) st.cp[a][k] = st.cp[a + 1][k];
          load_cp(t.n0 + t.step * step_rows, p, live, c + 16 * kAhead, nmax, st.cp[kAhead - 1], tma_out);
        }
        if (tma_out)
          finish(t.n0, p, live, c, min(16, nmax - c), v2 + 16 * h, cp, row, sm_g, sm_c, sm_h);
        else
          finish(t.n0 + t.step * step_rows, p, live, c, min(16, nmax - c), v2 + 16 * h, cp);
      }
      if (tma_out) {
        // this part's 32 batch rows are complete: its first thread stores
        // them while the part goes on with the next rows
        tc::fence_proxy_async_smem();
        tc::named_bar(2 + t.part, 128);
        if (threadIdx.x == 64 + 128 * t.part) {
          const int cx = CELL == LSTM ? t.m0 / 4 : t.m0, yb = t.n0 + c2, y0 = yb + t.step * step_rows;
          const bool fin = t.step == hT_step;
          if (write_gates) tc::tma_store_2d(&map_p, sm_g + (size_t)c2 * 128, t.m0, y0);
          if (CELL == LSTM) {
            tc::tma_store_2d(&map_c, sm_c + (size_t)c2 * kUnits, cx, y0);
            if (cT && fin) tc::tma_store_2d(&map_cT, sm_c + (size_t)c2 * kUnits, cx, yb);
          }
          tc::tma_store_2d(&map_h, sm_h + (size_t)c2 * kUnits, cx, y0);
          if (y) tc::tma_store_2d(&map_y, sm_h + (size_t)c2 * kUnits, cx, y0);
          if (hT && fin) tc::tma_store_2d(&map_hT, sm_h + (size_t)c2 * kUnits, cx, yb);
          tc::bulk_commit();
        }
      }
    }
    // the shared-memory tiles must outlive the stores' reads
    if (tma_out && threadIdx.x == 64 + 128 * t.part) {
      if (step_cnt) {
        // this part's stores of the step are complete and visible: the
        // pairs waiting to load h of this step may go on
        tc::bulk_wait_all();
        tc::fence_proxy_async_global();
        asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(step_cnt + t.step) : "memory");
      } else {
        tc::bulk_wait_read_all();
      }
    }
    // the part's next step reads this step's c (stored by its first thread)
    if (tma_out && step_cnt) tc::named_bar(2 + t.part, 128);
  }
};

// Forward LSTM step for CTAs that share their SM (one TMEM accumulator, three
// pipeline stages: a CTA of another launch fits beside it and streams its
// operands while this one runs its epilogue).  Tile = 128 packed gate rows x
// bn batch entries.  With no room to stage P in TMEM or whole output tiles
// in shared memory, each half of the epilogue warps walks its batch columns
// in slices of 16 through four slots of the freed pipeline buffers: a bulk
// tensor load brings the slice's P [16][128] into a slot three slices ahead
// of its use, the gates are activated in place, the cell update writes c and
// h beside them, and bulk tensor stores send the slot out while the next
// slices are computed.  The maps are those of the base with 16-row boxes.
template <int CELL>
struct EpiFwdStepTR : EpiFwdStepT<CELL> {
  static_assert(CELL == LSTM, "the shared-SM step is built for the LSTM cell");
  using Base = EpiFwdStepT<CELL>;
  using S = typename Base::S;
  static constexpr int kWarps = 8;
  static constexpr int kRows = 16;   // batch entries per slice
  static constexpr int kSlots = 4;   // per half of the epilogue warps
  static constexpr int kU = Base::kUnits;
  static constexpr int kSlotG = kRows * 128 * 4, kSlotC = kRows * kU * 4, kSlotH = kRows * kU * 2;
  static constexpr int kSlotBytes = kSlotG + kSlotC + kSlotH;
  static constexpr int kPartBytes = kSlots * kSlotBytes + 128;  // slots, then the slots' barriers
  int* err;
  uint64_t limit_ns;

  template <class Acc>
  __device__ __forceinline__ void operator()(const TileCoord& t, int row, const Acc& acc, int bn) const {
    const int H = this->H;
    const int p = t.m0 + row;
    const bool live = p < 4 * H;
    const int cw = bn / t.parts, cb = t.part * cw;
    const int nmax = min(cb + cw, this->B - t.n0);
    const int nsl = nmax > cb ? (nmax - cb + kRows - 1) / kRows : 0;
    uint8_t* ring = reinterpret_cast<uint8_t*>(t.red) + (size_t)t.part * kPartBytes;
    uint64_t* bar = reinterpret_cast<uint64_t*>(ring + kSlots * kSlotBytes);
    const bool leader = threadIdx.x == 64 + 128 * t.part;
    const int cx = t.m0 / 4;
    auto slot_g = [&](int k) { return reinterpret_cast<float*>(ring + (k & (kSlots - 1)) * kSlotBytes); };
    auto slot_c = [&](int k) { return reinterpret_cast<float*>(ring + (k & (kSlots - 1)) * kSlotBytes + kSlotG); };
    auto slot_h = [&](int k) { return reinterpret_cast<S*>(ring + (k & (kSlots - 1)) * kSlotBytes + kSlotG + kSlotC); };
    auto load_p = [&](int k) {
      tc::mbar_arrive_expect_tx(bar + (k & (kSlots - 1)), kSlotG);
      tc::tma_load_2d(slot_g(k), &this->map_p, bar + (k & (kSlots - 1)), t.m0, t.n0 + cb + kRows * k);
    };
    if (leader) {
      for (int i = 0; i < kSlots; ++i) tc::mbar_init(bar + i, 1);
      tc::fence_mbar_init();
      for (int k = 0; k < kSlots - 1 && k < nsl; ++k) load_p(k);
    }
    // c_{t-1} of the next kAhead chunks, in the lane mapping of the cell update
    constexpr int kAhead = Base::kAhead;
    float q[kAhead][4];
#pragma unroll
    for (int a = 0; a < kAhead; ++a) this->load_cp(t.n0, p, live, cb + kRows * a, nmax, q[a], true);
    tc::named_bar(2 + t.part, 128);  // the slots' barriers are initialised
    bool dead = false;
#pragma unroll 1
    for (int k = 0; k < nsl; ++k) {
      const int c = cb + kRows * k;
      float v[16], cp[4];
      acc.load16(c, v);
#pragma unroll
      for (int j = 0; j < 4; ++j) cp[j] = q[0][j];
#pragma unroll
      for (int a = 0; a + 1 < kAhead; ++a)
#pragma unroll
        for (int j = 0; j < 4; ++j) q[a][j] = q[a + 1][j];
      this->load_cp(t.n0, p, live, c + kRows * kAhead, nmax, q[kAhead - 1], true);
      if (!dead) {
        const uint64_t t0 = globaltimer_ns();
        while (!tc::mbar_try_wait(bar + (k & (kSlots - 1)), (uint32_t)((k / kSlots) & 1))) {
          if (globaltimer_ns() - t0 > limit_ns) {
            raise_error(err, DEV_TIMEOUT_PIPE);
            dead = true;
            break;
          }
        }
      }
      float* sg = slot_g(k);
#pragma unroll
      for (int i = 0; i < 16; ++i) v[i] += sg[i * 128 + row];
      this->finish(t.n0, p, live, 0, min(16, nmax - c), v, cp, row, sg, slot_c(k), slot_h(k));
      tc::fence_proxy_async_smem();
      tc::named_bar(2 + t.part, 128);
      if (leader) {
        const int y0 = t.n0 + c;
        if (this->write_gates) tc::tma_store_2d(&this->map_p, sg, t.m0, y0);
        tc::tma_store_2d(&this->map_c, slot_c(k), cx, y0);
        if (this->cT) tc::tma_store_2d(&this->map_cT, slot_c(k), cx, y0);
        tc::tma_store_2d(&this->map_h, slot_h(k), cx, y0);
        if (this->y) tc::tma_store_2d(&this->map_y, slot_h(k), cx, y0);
        if (this->hT) tc::tma_store_2d(&this->map_hT, slot_h(k), cx, y0);
        tc::bulk_commit();
        // slice k + 3 goes into the slot slice k - 1 was stored from
        if (k + kSlots - 1 < nsl) {
          tc::bulk_wait_read<1>();
          load_p(k + kSlots - 1);
        }
      }
    }
    // the slots must outlive the stores' reads
    if (leader) tc::bulk_wait_read_all();
  }
};

// Backward step product, tile = 128 hidden units x bn batch entries:
// acc[j][b] = (W_h^T dG_{s+1}^T)[j][b] = dh_s[b][j] before the gradient from
// above is added.  The epilogue only stores dh (fp32 [B][H]; bf16 dh0 for
// the final product); the pointwise step runs as its own full-occupancy
// kernel (bwd_point_v), whose wide loads keep far more bytes in flight than
// the epilogue threads of a CTA can.
//
// K splits run as one cluster per tile.  Their partial tiles meet through L2
// with bulk tensor copies: each CTA writes its partial, transposed to
// [batch][unit], into its (now idle) pipeline buffers, stores the slices
// other CTAs own to the partial-sum buffer, and after a cluster barrier loads
// the peers' partials of its own slice into the rows it just vacated, sums
// them in a fixed order and stores its slice of dh with one more bulk copy.
struct EpiBwdDhT {
  static constexpr int kWarps = 8;  // two warps per TMEM lane quadrant, each half of the columns
  using S = __nv_bfloat16;
  CUtensorMap map_part;  // partials [splits * Bp][H] fp32, box 128 units x (bn / splits) rows
  CUtensorMap map_dh;    // dh [B][H] fp32, same box
  // Fused LSTM pointwise step (fuse = 1; bn = 256 in clusters of 4): each CTA
  // runs it on its own 64-entry slice of dh while that is still in shared
  // memory, its inputs arriving by bulk loads of 16 batch rows at a time.
  CUtensorMap map_g;     // gates [B][4H] fp32, box 256 x 16 (64 units' four gates)
  CUtensorMap map_cs;    // c_s [B][H] fp32, box 128 x 16
  CUtensorMap map_cp;    // c_{s-1}, same (has_cp)
  CUtensorMap map_dc;    // carry, same
  CUtensorMap map_dy;    // dy [B][H] fp32 or bf16, box 128 x 16 (has_dy)
  int fuse, has_cp, has_dy, dy_f32;
  float* carry;          // [B][H] dc into step s (in) / into s-1 (out)
  float* dc0;            // [B][H] copy of the outgoing carry (s = 0), or null
  S* dGx;                // [B][4H]
  int B, H, Bp;          // Bp: batch rows per split in the partial buffer (a multiple of bn)
  float* dh;   // [B][H] (not final)
  S* dh0;      // [B][H] (final)
  int final_;
  int* err;
  uint64_t limit_ns;
  // inputs of the pointwise kernel that follows, pulled into L2 near the end
  // of the mainloop (null: none)
  const float* pf_gates;  // [B][G*H]
  const float* pf_c_s;    // [B][H]
  const float* pf_c_sm1;  // [B][H]
  int G;

  __device__ __forceinline__ void prefetch(const TileCoord&, int, int) const {}

  // this CTA's (unit, batch entry) block of the pointwise inputs
  __device__ __forceinline__ void tail_prefetch(const TileCoord& t, int bn) const {
    if (!pf_gates || t.m0 >= H) return;
    const int cw = t.cluster > 1 ? bn / t.cluster : bn;
    const int b0 = t.n0 + (t.cluster > 1 ? t.split * cw : 0);
    const int units = min(128, H - t.m0);
    for (int i = 0; i < cw; ++i) {
      const int b = b0 + i;
      if (b >= B) break;
      tc::prefetch_l2(pf_gates + (size_t)b * G * H + (size_t)G * t.m0, units * G * 4);
      if (pf_c_s) tc::prefetch_l2(pf_c_s + (size_t)b * H + t.m0, units * 4);
      if (pf_c_sm1) tc::prefetch_l2(pf_c_sm1 + (size_t)b * H + t.m0, units * 4);
    }
  }

  // Shared-memory home of one 16-row quarter of the pointwise inputs.
  struct Quarter {
    float* g;   // [2][16][256]: gates of units 0-63, then 64-127 (the two bulk boxes)
    float* cs;  // [16][128]
    float* cp;
    float* dc;
    void* dy;   // [16][128] fp32 or bf16
  };
  __device__ __forceinline__ uint32_t quarter_bytes() const {
    return 32768u + 8192u * (2u + (has_cp ? 1u : 0u)) + (has_dy ? (dy_f32 ? 8192u : 4096u) : 0u);
  }
  __device__ __forceinline__ void load_quarter(const Quarter& qd, uint64_t* bar, int m0, int b) const {
    tc::mbar_arrive_expect_tx(bar, quarter_bytes());
    tc::tma_load_2d(qd.g, &map_g, bar, 4 * m0, b);
    tc::tma_load_2d(qd.g + 16 * 256, &map_g, bar, 4 * m0 + 256, b);
    tc::tma_load_2d(qd.cs, &map_cs, bar, m0, b);
    if (has_cp) tc::tma_load_2d(qd.cp, &map_cp, bar, m0, b);
    tc::tma_load_2d(qd.dc, &map_dc, bar, m0, b);
    if (has_dy) tc::tma_load_2d(qd.dy, &map_dy, bar, m0, b);
  }
  // the pointwise step for rows [r0, r0 + 8) of a quarter starting at batch entry b0
  __device__ __forceinline__ void run_quarter(const Quarter& qd, const float* dh_rows, int row, int j, bool live,
                                              int b0, int r0) const {
    const float4* g4 = reinterpret_cast<const float4*>(qd.g + (row >> 6) * 16 * 256) + (row & 63);
#pragma unroll 4
    for (int r = r0; r < r0 + 8; ++r) {
      const int b = b0 + r;
      if (!live || b >= B) continue;
      float dh = dh_rows[r * 128 + row];
      if (has_dy)
        dh += dy_f32 ? static_cast<const float*>(qd.dy)[r * 128 + row]
                     : __bfloat162float(static_cast<const S*>(qd.dy)[r * 128 + row]);
      const float4 gt = g4[r * 64];
      const float cs = qd.cs[r * 128 + row], cp = has_cp ? qd.cp[r * 128 + row] : 0.f, dc = qd.dc[r * 128 + row];
      const float tau = tanh_hw(cs);
      const float dov = dh * tau;
      const float dcv = dc + dh * gt.w * (1.f - tau * tau);
      const float d0 = dcv * gt.z * gt.x * (1.f - gt.x);
      const float d1 = dcv * cp * gt.y * (1.f - gt.y);
      const float d2 = dcv * gt.x * (1.f - gt.z * gt.z);
      const float d3 = dov * gt.w * (1.f - gt.w);
      const size_t bj = (size_t)b * H + j;
      carry[bj] = dcv * gt.y;
      if (dc0) dc0[bj] = dcv * gt.y;
      *reinterpret_cast<uint2*>(dGx + (size_t)b * 4 * H + 4 * (size_t)j) = make_uint2(pack_bf16x2(d0, d1), pack_bf16x2(d2, d3));
    }
  }

  __device__ __forceinline__ void put(int j, int b, float v) const {
    const size_t bj = (size_t)b * H + j;
    if (final_) dh0[bj] = __float2bfloat16_rn(v);
    else dh[bj] = v;
  }

  template <class Acc>
  __device__ __forceinline__ void operator()(const TileCoord& t, int row, const Acc& acc, int bn) const {
    const int j = t.m0 + row;
    const bool live = j < H && (!final_ || dh0);
    const int lane = threadIdx.x & 31;
    if (t.cluster > 1) {
      constexpr int EWT = kWarps * 32;
      const bool leader = threadIdx.x == 64;  // first epilogue thread
      const int cw = bn / t.cluster;
      float* tile = t.red;  // [bn][128]: tile[b * 128 + row]
      // fused pointwise: quarters 0 and 2 go to the pipeline buffers past the
      // tile (region A), quarters 1 and 3 to two slices other CTAs own (region B)
      const bool fz = fuse && !final_ && bn == 256 && t.cluster == 4;
      const int b_own = t.n0 + t.split * cw;
      Quarter qa, qb;
      {
        float* ra = tile + (size_t)bn * 128;
        qa = Quarter{ra, ra + 8192, ra + 10240, ra + 12288, ra + 14336};
        const int o1 = t.split == 0 ? 1 : 0, o2 = t.split <= 1 ? 2 : 1;
        float* s1 = tile + (size_t)o1 * cw * 128;
        float* s2 = tile + (size_t)o2 * cw * 128;
        qb = Quarter{s1, s2, s2 + 2048, s2 + 4096, s2 + 6144};
      }
      if (fz && leader) load_quarter(qa, t.aux + 1, t.m0, b_own);
      // 1. partial tile -> shared memory as [batch][unit]
      for (int c = t.part * (bn / t.parts); c < (t.part + 1) * (bn / t.parts); c += 16) {
        float v[16];
        acc.load16(c, v);
#pragma unroll
        for (int i = 0; i < 16; ++i) tile[(c + i) * 128 + row] = v[i];
      }
      tc::fence_proxy_async_smem();
      tc::named_bar(1, EWT);
      // 2. the slices other CTAs own go to the partial buffer (rows split*Bp + batch)
      if (leader) {
        for (int o = 0; o < t.cluster; ++o)
          if (o != t.split) tc::tma_store_2d(&map_part, tile + (size_t)o * cw * 128, t.m0, t.split * Bp + t.n0 + o * cw);
        tc::bulk_commit();
        tc::bulk_wait_all();
        tc::fence_proxy_async_global();
      }
      tc::named_bar(1, EWT);
      const uint32_t full_local = tc::smem_addr(t.red_full);
      __syncwarp();
      if (lane == 0)
        for (int p = 0; p < t.cluster; ++p) tc::mbar_arrive_remote(tc::mapa(full_local, t.peer_base + p * t.peer_stride));
      int ok = 1;
      if (lane == 0) ok = tc::mbar_wait_cluster(t.red_full, 0, err, limit_ns) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      // 3. the peers' partials of this CTA's slice, into the rows they vacated
      if (leader && ok) {
        tc::fence_proxy_async_global();
        tc::mbar_arrive_expect_tx(t.aux, (uint32_t)((t.cluster - 1) * cw * 128 * 4));
        for (int sp = 0; sp < t.cluster; ++sp)
          if (sp != t.split)
            tc::tma_load_2d(tile + (size_t)sp * cw * 128, &map_part, t.aux, t.m0, sp * Bp + t.n0 + t.split * cw);
      }
      if (lane == 0 && ok) ok = tc::mbar_wait_cluster(t.aux, 0, err, limit_ns) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      // 4. own slice = own partial + peers' partials in split order; dh by one bulk store.
      // Partial sp of this slice's batch row r sits at tile row sp * cw + r for
      // every sp (the own partial included), so the sum runs over contiguous
      // 16-byte vectors, with no tie to the TMEM lane a thread was given.
      if (ok && !final_) {
        const int et = threadIdx.x - 64;  // epilogue threads are 64 .. 64 + EWT - 1
        const float4* t4 = reinterpret_cast<const float4*>(tile);
        float4* o4 = reinterpret_cast<float4*>(tile) + (size_t)t.split * cw * 32;
#pragma unroll 2
        for (int f = et; f < cw * 32; f += EWT) {
          float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int sp = 0; sp < 8; ++sp) {
            if (sp < t.cluster) {
              const float4 w = t4[(size_t)sp * cw * 32 + f];
              v.x += w.x;
              v.y += w.y;
              v.z += w.z;
              v.w += w.w;
            }
          }
          o4[f] = v;
        }
      } else if (ok) {
        // final product (dh0 in the storage type): 8 rows at a time, every
        // partial's loads issued before the adds
        const int pw = cw / t.parts;  // a multiple of 8
        const int r0 = t.split * cw + t.part * pw;
#pragma unroll 1
        for (int r = r0; r < r0 + pw; r += 8) {
          float v[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) v[i] = 0.f;
#pragma unroll
          for (int sp = 0; sp < 8; ++sp) {
            if (sp < t.cluster) {
              const float* src = tile + (size_t)(sp == t.split ? r : sp * cw + (r - t.split * cw)) * 128 + row;
              float w[8];
#pragma unroll
              for (int i = 0; i < 8; ++i) w[i] = src[i * 128];
#pragma unroll
              for (int i = 0; i < 8; ++i) v[i] += w[i];
            }
          }
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            if (final_) {
              if (live && t.n0 + r + i < B) put(j, t.n0 + r + i, v[i]);
            } else {
              tile[(size_t)(r + i) * 128 + row] = v[i];
            }
          }
        }
      }
      if (fz) {
        // 5. the pointwise step on the own slice, 16 batch rows per bulk load
        const float* dh_rows = tile + (size_t)t.split * cw * 128;
        const int r0 = t.part * 8;
        tc::fence_proxy_async_smem();
        tc::named_bar(1, EWT);  // the peers' partials in region B have been read
        if (leader && ok) load_quarter(qb, t.aux + 2, t.m0, b_own + 16);
        for (int q = 0; q < 4; ++q) {
          const Quarter& qd = (q & 1) ? qb : qa;
          uint64_t* bar = t.aux + 1 + (q & 1);
          if (lane == 0 && ok) ok = tc::mbar_wait_cluster(bar, (uint32_t)(q >> 1), err, limit_ns) ? 1 : 0;
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (ok) run_quarter(qd, dh_rows + (size_t)16 * q * 128, row, j, live, b_own + 16 * q, r0);
          if (q < 2) {
            // reload this region with quarter q + 2 once every thread is done with it
            tc::fence_proxy_async_smem();
            tc::named_bar(1, EWT);
            if (leader && ok) load_quarter(qd, bar, t.m0, b_own + 16 * (q + 2));
          }
        }
      } else if (!final_) {
        tc::fence_proxy_async_smem();
        tc::named_bar(1, EWT);
        if (leader && ok) {
          tc::tma_store_2d(&map_dh, tile + (size_t)t.split * cw * 128, t.m0, t.n0 + t.split * cw);
          tc::bulk_commit();
          tc::bulk_wait_read_all();
        }
      }
      if (!ok && leader) {
        // loads may still be landing in this CTA's buffers: let them (bounded)
        const uint64_t t0 = globaltimer_ns();
        while (!tc::mbar_try_wait(t.aux, 0) && globaltimer_ns() - t0 < 1000000ull) {
        }
        if (fz)
          for (int a = 1; a < 3; ++a)
            for (int ph = 0; ph < 2; ++ph)
              while (!tc::mbar_try_wait(t.aux + a, ph) && globaltimer_ns() - t0 < 2000000ull) {
              }
      }
      return;
    }
    const int pw = bn / t.parts;
    const int nmax = min((t.part + 1) * pw, B - t.n0);
    for (int c = t.part * pw; c < nmax; c += 16) {
      float v[16];
      acc.load16(c, v);
      const int nb = min(16, nmax - c);
      if (live) {
#pragma unroll
        for (int i = 0; i < 16; ++i)
          if (i < nb) put(j, t.n0 + c + i, v[i]);
      }
    }
  }
};

// Pointwise backward step s for the packing unit 1, four hidden units of one
// batch entry per thread (16-byte loads and stores throughout):
//   dh = dh_s (+ dy_s);  LSTM: tau = tanh(c_s), dc = carry + dh o (1 - tau^2),
//   d(i, f, g, o) = (dc g i(1-i), dc c_{s-1} f(1-f), dc i (1-g^2), dh tau o(1-o)),
//   carry <- dc f;   tanh RNN: d = dh (1 - h_s^2).
template <int CELL>
struct BwdPointV {
  using S = __nv_bfloat16;
  int B, H;
  const float* dh;      // [B][H] product part of dh_s, or null
  const S* dh_init;     // [B][H] used when dh is null (gradient into the last step), or null = zero
  const void* dy;       // [B][H] (float if dy_f32 else S), or null
  int dy_f32;
  const float* gates;   // [B][G*H] activated gates of step s (tanh RNN: h_s)
  const float* c_s;     // LSTM [B][H]
  const float* c_sm1;   // LSTM [B][H], null = zero
  float* carry;         // LSTM [B][H]: dc into step s (in) / into s-1 (out)
  float* dc0;           // LSTM [B][H]: also receives the outgoing carry (s = 0), or null
  S* dGx;               // [B][G*H]

  __device__ __forceinline__ void run(long long q) const {
    // q indexes groups of four hidden units: b = q / (H/4), j0 = 4 (q % (H/4))
    const int hq = H / 4;
    const int b = (int)(q / hq), j0 = 4 * (int)(q % hq);
    const size_t bj = (size_t)b * H + j0;
    float4 d = dh ? *reinterpret_cast<const float4*>(dh + bj) : make_float4(0.f, 0.f, 0.f, 0.f);
    if (!dh && dh_init) {
      const uint2 w = *reinterpret_cast<const uint2*>(dh_init + bj);
      d = make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xFFFF0000u), __uint_as_float(w.y << 16),
                      __uint_as_float(w.y & 0xFFFF0000u));
    }
    if (dy) {
      if (dy_f32) {
        const float4 e = *reinterpret_cast<const float4*>(static_cast<const float*>(dy) + bj);
        d.x += e.x; d.y += e.y; d.z += e.z; d.w += e.w;
      } else {
        const uint2 w = *reinterpret_cast<const uint2*>(static_cast<const S*>(dy) + bj);
        d.x += __uint_as_float(w.x << 16); d.y += __uint_as_float(w.x & 0xFFFF0000u);
        d.z += __uint_as_float(w.y << 16); d.w += __uint_as_float(w.y & 0xFFFF0000u);
      }
    }
    const float dhv[4] = {d.x, d.y, d.z, d.w};
    if constexpr (CELL == LSTM) {
      const float4* gp = reinterpret_cast<const float4*>(gates + (size_t)b * 4 * H + 4 * (size_t)j0);
      const float4 g4[4] = {gp[0], gp[1], gp[2], gp[3]};
      const float4 cs = *reinterpret_cast<const float4*>(c_s + bj);
      const float4 cp = c_sm1 ? *reinterpret_cast<const float4*>(c_sm1 + bj) : make_float4(0.f, 0.f, 0.f, 0.f);
      const float4 dc = *reinterpret_cast<const float4*>(carry + bj);
      const float csv[4] = {cs.x, cs.y, cs.z, cs.w}, cpv[4] = {cp.x, cp.y, cp.z, cp.w}, dcv_in[4] = {dc.x, dc.y, dc.z, dc.w};
      float dco[4];
      uint32_t packed[8];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float4 gt = g4[k];
        const float tau = tanh_hw(csv[k]);
        const float dov = dhv[k] * tau;
        const float dcv = dcv_in[k] + dhv[k] * gt.w * (1.f - tau * tau);
        const float d0 = dcv * gt.z * gt.x * (1.f - gt.x);
        const float d1 = dcv * cpv[k] * gt.y * (1.f - gt.y);
        const float d2 = dcv * gt.x * (1.f - gt.z * gt.z);
        const float d3 = dov * gt.w * (1.f - gt.w);
        dco[k] = dcv * gt.y;
        packed[2 * k] = pack_bf16x2(d0, d1);
        packed[2 * k + 1] = pack_bf16x2(d2, d3);
      }
      const float4 co = make_float4(dco[0], dco[1], dco[2], dco[3]);
      *reinterpret_cast<float4*>(carry + bj) = co;
      if (dc0) *reinterpret_cast<float4*>(dc0 + bj) = co;
      uint4* gx = reinterpret_cast<uint4*>(dGx + (size_t)b * 4 * H + 4 * (size_t)j0);
      gx[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
      gx[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
    } else {
      const float4 hv = *reinterpret_cast<const float4*>(gates + bj);
      const float hvv[4] = {hv.x, hv.y, hv.z, hv.w};
      float o[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) o[k] = dhv[k] * simple_slope<CELL>(hvv[k]);
      *reinterpret_cast<uint2*>(dGx + bj) = make_uint2(pack_bf16x2(o[0], o[1]), pack_bf16x2(o[2], o[3]));
    }
  }
};

}  // namespace rnn
