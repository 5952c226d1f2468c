// rnn_ref.cpp -- plain double-precision oracle for stacked LSTM / GRU / simple RNN.
//
// TEST INFRASTRUCTURE ONLY: used by the tests, the smoke check and the
// benchmark's CPU-baseline leg; never by the product library.
//
// Source of the method: "Optimizing Performance of Recurrent Neural Networks
// on GPUs" (review page, section "제안 방법"): LSTM groups four gate matrices,
// GRU three, the simple RNN one; the weight update is one product over all
// timesteps with a negligible bias update.  The pages give no equations, so the
// cells below are the textbook definitions:
//   LSTM (gates i,f,g,o):  a = W_x in + b_x + W_h h + b_h
//        i=s(a_i) f=s(a_f) g=tanh(a_g) o=s(a_o); c'=f c+i g; h'=o tanh(c')
//   GRU (gates r,z,n):     r=s(x_r+h_r) z=s(x_z+h_z) n=tanh(x_n + r*h_n)
//        with x_* = W_x in + b_x, h_* = W_h h + b_h;  h' = (1-z) n + z h
//   RNN:                   h' = tanh(W_x in + b_x + W_h h + b_h)
//   ReLU RNN:              h' = max(0, W_x in + b_x + W_h h + b_h)
// Variable lengths (the *_len entry points): sequence b runs steps
// 0 .. lens[b]-1; afterwards its outputs are 0 and its state is carried, so
// hT / cT are its state after its own last step.
// Bidirectional layers (the *_dir entry points, D = 2): every layer has a
// second set of weights that runs the same cell over time in reverse (from
// t = T-1, or from t = lens[b]-1, down to 0, starting from its own h0); the
// layer's output at t is [h_forward(t), h_reverse(t)] and feeds the next
// layer.  Each (layer, direction) is kept in its own step order: step s is
// time s forward and time T-1-s in reverse, so in reverse a shorter
// sequence's idle steps come first and carry h0 until its last time.
// The backward pass is the exact gradient of
//   L = sum(y*dy) + sum(hT*dhT) + sum(cT*dcT)
// taken in reverse time, top layer first, one step and one layer at a time
// (no reordering beyond the definition).
// ReLU decisions in a given precision (the *_kp entry points): the on/off
// decision a > 0 of the ReLU cell is a comparison of a floating-point value,
// and a device that stores h in bf16 or fp32 can take it differently from
// double arithmetic where a is close to 0.  With decide = 1 (bf16) or 2 (fp32)
// the decisions come from a first forward pass whose h is rounded to that
// type after every step (round to nearest even, as the device stores it);
// with decide = 3 they are given by the caller.  Every value, forward and
// backward, is then computed in double with those decisions imposed (h = a
// where on, 0 where off; slope 1 where on).
#include "rnn_ref.h"

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>
#ifdef _OPENMP
#include <omp.h>
#endif

namespace {

struct LayerW {
  const double* Wx;
  const double* Wh;
  const double* bx;
  const double* bh;
  int In;
};

int gates_of(int cell) { return cell == RNN_REF_LSTM ? 4 : (cell == RNN_REF_GRU ? 3 : 1); }

double sigm(double a) { return 1.0 / (1.0 + std::exp(-a)); }

// one entry per (layer, direction) v = l * D + d; the input of layer l >= 1
// is the D * H wide output of layer l - 1
std::vector<LayerW> split_weights(const double* w, int G, int L, int D, int I, int H) {
  std::vector<LayerW> v((size_t)L * D);
  const double* p = w;
  for (int l = 0; l < L; ++l) {
    for (int d = 0; d < D; ++d) {
      LayerW& e = v[(size_t)l * D + d];
      const int In = l == 0 ? I : D * H;
      e.In = In;
      e.Wx = p; p += (size_t)G * H * In;
      e.Wh = p; p += (size_t)G * H * H;
      e.bx = p; p += (size_t)G * H;
      e.bh = p; p += (size_t)G * H;
    }
  }
  return v;
}

// time of step s in direction d, and whether sequence b runs it
inline int time_of(int d, int T, int s) { return d == 0 ? s : T - 1 - s; }
inline bool runs(const int* lens, int b, int t) { return !lens || t < lens[b]; }

// Everything the backward pass needs from the forward pass, per (layer,
// direction), indexed by step s (time_of(d, T, s)).
struct Record {
  int T, B, H, G;
  std::vector<double> hs;     // (T+1) x B x H, slot 0 = h0, slot s+1 = h after step s
  std::vector<double> cs;     // (T+1) x B x H (LSTM)
  std::vector<double> gates;  // T x B x G*H   activated gate values
  std::vector<double> hn;     // T x B x H     GRU: W_hn h_prev + b_hn
  std::vector<unsigned char> on;  // T x B x H ReLU: the on/off decision of each unit
  double* h(int t1, int b) { return &hs[((size_t)t1 * B + b) * H]; }
  double* c(int t1, int b) { return &cs[((size_t)t1 * B + b) * H]; }
  double* g(int t, int b) { return &gates[((size_t)t * B + b) * G * H]; }
  double* n(int t, int b) { return &hn[((size_t)t * B + b) * H]; }
  unsigned char* o(int t, int b) { return &on[((size_t)t * B + b) * H]; }
};

// v rounded as the device stores it: 1 = bf16 (via float, then to nearest
// even on the upper 16 bits of the float), 2 = float; 0 = unchanged.
double store_round(double v, int prec) {
  if (prec == 0) return v;
  float f = (float)v;
  if (prec == 1) {
    uint32_t u;
    std::memcpy(&u, &f, 4);
    if ((u & 0x7F800000u) != 0x7F800000u) u = (u + 0x7FFFu + ((u >> 16) & 1u)) & 0xFFFF0000u;
    std::memcpy(&f, &u, 4);
  }
  return (double)f;
}

bool bad_args(int cell, int L, int D, int T, int B, int I, int H, const double* x, const double* w) {
  return cell < 0 || cell > 3 || L < 1 || D < 1 || D > 2 || T < 0 || B < 0 || I < 1 || H < 1 ||
         (!x && T * B > 0) || !w;
}

// Forward over all layers; fills one Record per (layer, direction) and the
// layer outputs out[l] = [T][B][D*H] (zero where a sequence has ended).
// lens (nullable = all T): sequence b runs times 0 .. lens[b]-1; at its other
// steps its state is carried unchanged (so slot T holds its final state).
// round_h: h stored rounded (store_round) after every step; relu_in (nullable):
// ReLU decisions to impose, one vector per (layer, direction), T x B x H.
// preact (nullable): ReLU pre-activations [L*D][T][B][H] by step.
void forward(int cell, int L, int D, int T, int B, int I, int H, const double* x, const double* h0,
             const double* c0, const std::vector<LayerW>& W, std::vector<Record>& rec,
             std::vector<std::vector<double>>& out, const int* lens, int round_h = 0,
             const std::vector<std::vector<unsigned char>>* relu_in = nullptr,
             std::vector<double>* preact = nullptr) {
  if (preact) preact->assign((size_t)L * D * T * B * H, 0.0);
  const int G = gates_of(cell);
  const int GH = G * H, DH = D * H;
  rec.assign((size_t)L * D, Record());
  out.assign(L, std::vector<double>());
  for (int l = 0; l < L; ++l) {
    out[l].assign((size_t)T * B * DH, 0.0);
    for (int d = 0; d < D; ++d) {
      const int v = l * D + d;
      Record& R = rec[v];
      R.T = T; R.B = B; R.H = H; R.G = G;
      R.hs.assign((size_t)(T + 1) * B * H, 0.0);
      R.gates.assign((size_t)T * B * GH, 0.0);
      if (cell == RNN_REF_LSTM) R.cs.assign((size_t)(T + 1) * B * H, 0.0);
      if (cell == RNN_REF_GRU) R.hn.assign((size_t)T * B * H, 0.0);
      if (cell == RNN_REF_RELU) R.on.assign((size_t)T * B * H, 0);
      if (h0) std::memcpy(R.h(0, 0), h0 + (size_t)v * B * H, sizeof(double) * B * H);
      if (c0 && cell == RNN_REF_LSTM) std::memcpy(R.c(0, 0), c0 + (size_t)v * B * H, sizeof(double) * B * H);
      const LayerW& lw = W[v];
      std::vector<double> ax((size_t)B * GH), ah((size_t)B * GH);
      for (int st = 0; st < T; ++st) {
        const int t = time_of(d, T, st);
        // pre-activations: one dot product per (batch row, gate row)
#pragma omp parallel for collapse(2) schedule(static)
        for (int b = 0; b < B; ++b) {
          for (int p = 0; p < GH; ++p) {
            const double* in = l == 0 ? x + ((size_t)t * B + b) * I : &out[l - 1][((size_t)t * B + b) * DH];
            const double* hp = R.h(st, b);
            const double* wx = lw.Wx + (size_t)p * lw.In;
            const double* wh = lw.Wh + (size_t)p * H;
            double sx = lw.bx[p], sh = lw.bh[p];
            for (int k = 0; k < lw.In; ++k) sx += wx[k] * in[k];
            for (int k = 0; k < H; ++k) sh += wh[k] * hp[k];
            ax[(size_t)b * GH + p] = sx;
            ah[(size_t)b * GH + p] = sh;
          }
        }
        // pointwise cell update
#pragma omp parallel for collapse(2) schedule(static)
        for (int b = 0; b < B; ++b) {
          for (int j = 0; j < H; ++j) {
            const double* sx = &ax[(size_t)b * GH];
            const double* sh = &ah[(size_t)b * GH];
            double* gt = R.g(st, b);
            double hprev = R.h(st, b)[j];
            double hnew;
            if (!runs(lens, b, t)) {
              // idle step of this sequence: state carried, no gate values, output 0
              R.h(st + 1, b)[j] = hprev;
              if (cell == RNN_REF_LSTM) R.c(st + 1, b)[j] = R.c(st, b)[j];
              continue;
            }
            if (cell == RNN_REF_LSTM) {
              double i = sigm(sx[j] + sh[j]);
              double f = sigm(sx[H + j] + sh[H + j]);
              double g = std::tanh(sx[2 * H + j] + sh[2 * H + j]);
              double o = sigm(sx[3 * H + j] + sh[3 * H + j]);
              double c = f * R.c(st, b)[j] + i * g;
              hnew = o * std::tanh(c);
              R.c(st + 1, b)[j] = c;
              gt[j] = i; gt[H + j] = f; gt[2 * H + j] = g; gt[3 * H + j] = o;
            } else if (cell == RNN_REF_GRU) {
              double r = sigm(sx[j] + sh[j]);
              double z = sigm(sx[H + j] + sh[H + j]);
              double hn = sh[2 * H + j];
              double n = std::tanh(sx[2 * H + j] + r * hn);
              hnew = (1.0 - z) * n + z * hprev;
              R.n(st, b)[j] = hn;
              gt[j] = r; gt[H + j] = z; gt[2 * H + j] = n;
            } else if (cell == RNN_REF_RELU) {
              const double a = sx[j] + sh[j];
              const bool on = relu_in ? (*relu_in)[v][((size_t)st * B + b) * H + j] != 0 : a > 0.0;
              if (preact) (*preact)[(((size_t)v * T + st) * B + b) * H + j] = a;
              R.o(st, b)[j] = on ? 1 : 0;
              hnew = on ? a : 0.0;
              gt[j] = hnew;
            } else {
              hnew = std::tanh(sx[j] + sh[j]);
              gt[j] = hnew;
            }
            hnew = store_round(hnew, round_h);
            R.h(st + 1, b)[j] = hnew;
            out[l][((size_t)t * B + b) * DH + (size_t)d * H + j] = hnew;
          }
        }
      }
    }
  }
}

// The forward pass with ReLU decisions taken in precision `decide` (see the
// header comment): a first pass with h rounded after every step records the
// decisions, a second exact pass imposes them.  Other cells, or decide = 0:
// one exact pass.
// on (nullable, [L*D][T][B][H] by time): the decisions given (decide = 3) or
// taken; preact (nullable, same layout): the ReLU pre-activations of the pass
// that took them.
void forward_kp(int cell, int L, int D, int T, int B, int I, int H, const double* x, const double* h0,
                const double* c0, const std::vector<LayerW>& W, std::vector<Record>& rec,
                std::vector<std::vector<double>>& out, const int* lens, int decide, unsigned char* on_io,
                double* preact) {
  const size_t per = (size_t)T * B * H;
  auto by_time = [&](int v, int st) { return (size_t)v * per + (size_t)time_of(v % D, T, st) * B * H; };
  if (cell != RNN_REF_RELU) {
    forward(cell, L, D, T, B, I, H, x, h0, c0, W, rec, out, lens);
    return;
  }
  std::vector<std::vector<unsigned char>> on(rec.size());
  if (decide == 3) {
    on.assign((size_t)L * D, std::vector<unsigned char>(per));
    for (int v = 0; v < L * D; ++v)
      for (int st = 0; st < T; ++st)
        std::memcpy(&on[v][(size_t)st * B * H], on_io + by_time(v, st), (size_t)B * H);
  } else {
    std::vector<double> pre;
    forward(cell, L, D, T, B, I, H, x, h0, c0, W, rec, out, lens, decide, nullptr, preact ? &pre : nullptr);
    on.resize(rec.size());
    for (size_t v = 0; v < rec.size(); ++v) on[v] = rec[v].on;
    for (int v = 0; v < L * D; ++v)
      for (int st = 0; st < T; ++st) {
        if (on_io) std::memcpy(on_io + by_time(v, st), &on[v][(size_t)st * B * H], (size_t)B * H);
        if (preact) std::memcpy(preact + by_time(v, st), &pre[(size_t)v * per + (size_t)st * B * H],
                                sizeof(double) * B * H);
      }
    if (decide == 0) return;  // the decisions are the double ones: this pass is the result
  }
  forward(cell, L, D, T, B, I, H, x, h0, c0, W, rec, out, lens, 0, &on);
}

bool bad_lens(int T, int B, const int* lens) {
  if (!lens) return false;
  for (int b = 0; b < B; ++b)
    if (lens[b] < 0 || lens[b] > T) return true;
  return false;
}

}  // namespace

extern "C" int rnn_ref_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

extern "C" int rnn_ref_fwd_kp(int cell, int L, int D, int T, int B, int I, int H, const int* lens, int decide,
                              unsigned char* on, double* preact, const double* x, const double* h0,
                              const double* c0, const double* w, double* y, double* hT, double* cT) {
  if (bad_args(cell, L, D, T, B, I, H, x, w) || bad_lens(T, B, lens) || decide < 0 || decide > 3 ||
      (decide == 3 && !on))
    return -1;
  const int G = gates_of(cell);
  std::vector<LayerW> W = split_weights(w, G, L, D, I, H);
  std::vector<Record> rec;
  std::vector<std::vector<double>> out;
  forward_kp(cell, L, D, T, B, I, H, x, h0, c0, W, rec, out, lens, decide, on, preact);
  if (y && T > 0) std::memcpy(y, out[L - 1].data(), sizeof(double) * (size_t)T * B * D * H);
  for (int v = 0; v < L * D; ++v) {
    if (hT) std::memcpy(hT + (size_t)v * B * H, rec[v].h(T, 0), sizeof(double) * B * H);
    if (cT && cell == RNN_REF_LSTM)
      std::memcpy(cT + (size_t)v * B * H, rec[v].c(T, 0), sizeof(double) * B * H);
  }
  return 0;
}

extern "C" int rnn_ref_fwd_dir(int cell, int L, int D, int T, int B, int I, int H, const int* lens,
                               const double* x, const double* h0, const double* c0, const double* w, double* y,
                               double* hT, double* cT) {
  return rnn_ref_fwd_kp(cell, L, D, T, B, I, H, lens, 0, nullptr, nullptr, x, h0, c0, w, y, hT, cT);
}

extern "C" int rnn_ref_fwd_len(int cell, int L, int T, int B, int I, int H, const int* lens, const double* x,
                               const double* h0, const double* c0, const double* w, double* y,
                               double* hT, double* cT) {
  return rnn_ref_fwd_dir(cell, L, 1, T, B, I, H, lens, x, h0, c0, w, y, hT, cT);
}

extern "C" int rnn_ref_fwd(int cell, int L, int T, int B, int I, int H, const double* x,
                           const double* h0, const double* c0, const double* w, double* y,
                           double* hT, double* cT) {
  return rnn_ref_fwd_dir(cell, L, 1, T, B, I, H, nullptr, x, h0, c0, w, y, hT, cT);
}

extern "C" int rnn_ref_bwd_kp(int cell, int L, int D, int T, int B, int I, int H, const int* lens, int decide,
                              unsigned char* on, const double* x, const double* h0, const double* c0,
                              const double* w, const double* dy, const double* dhT, const double* dcT, double* dx,
                              double* dh0, double* dc0, double* dw) {
  if (bad_args(cell, L, D, T, B, I, H, x, w) || (!dy && T * B > 0) || bad_lens(T, B, lens) || decide < 0 ||
      decide > 3 || (decide == 3 && !on))
    return -1;
  const int G = gates_of(cell);
  const int GH = G * H, DH = D * H;
  std::vector<LayerW> W = split_weights(w, G, L, D, I, H);
  std::vector<Record> rec;
  std::vector<std::vector<double>> out;
  forward_kp(cell, L, D, T, B, I, H, x, h0, c0, W, rec, out, lens, decide, on, nullptr);

  // gradient arriving at each layer's outputs [T][B][D*H] from above (dy for the top layer)
  std::vector<double> dabove(dy, dy + (size_t)T * B * DH);
  // weight-gradient views into dw (same layout as w), zeroed first
  struct LayerDW { double *Wx, *Wh, *bx, *bh; };
  std::vector<LayerDW> dW((size_t)L * D);
  if (dw) {
    double* p = dw;
    for (int v = 0; v < L * D; ++v) {
      dW[v].Wx = p; p += (size_t)GH * W[v].In;
      dW[v].Wh = p; p += (size_t)GH * H;
      dW[v].bx = p; p += GH;
      dW[v].bh = p; p += GH;
    }
    std::memset(dw, 0, sizeof(double) * (size_t)(p - dw));
  }

  for (int l = L - 1; l >= 0; --l) {
    const int In = l == 0 ? I : DH;
    std::vector<double> dbelow((size_t)T * B * In, 0.0);  // gradient wrt this layer's inputs, both directions
    for (int d = 0; d < D; ++d) {
      const int v = l * D + d;
      Record& R = rec[v];
      const LayerW& lw = W[v];
      std::vector<double> dh_rec((size_t)B * H, 0.0), dc_rec((size_t)B * H, 0.0);
      if (dhT) std::memcpy(dh_rec.data(), dhT + (size_t)v * B * H, sizeof(double) * B * H);
      if (dcT && cell == RNN_REF_LSTM) std::memcpy(dc_rec.data(), dcT + (size_t)v * B * H, sizeof(double) * B * H);
      std::vector<double> dGx((size_t)B * GH), dGh((size_t)B * GH);
      std::vector<double> dh_new((size_t)B * H), dc_new((size_t)B * H);

      for (int st = T - 1; st >= 0; --st) {
        const int t = time_of(d, T, st);
        // pointwise: gate pre-activation gradients of step st
#pragma omp parallel for collapse(2) schedule(static)
        for (int b = 0; b < B; ++b) {
          for (int j = 0; j < H; ++j) {
            const double* gt = R.g(st, b);
            double* gx = &dGx[(size_t)b * GH];
            double* gh = &dGh[(size_t)b * GH];
            if (!runs(lens, b, t)) {
              // idle step: the identity on the state with the constant output 0,
              // so the state gradient passes through
              for (int q = 0; q < G; ++q) gx[q * H + j] = gh[q * H + j] = 0.0;
              dh_new[(size_t)b * H + j] = dh_rec[(size_t)b * H + j];
              if (cell == RNN_REF_LSTM) dc_new[(size_t)b * H + j] = dc_rec[(size_t)b * H + j];
              continue;
            }
            double dh = dabove[((size_t)t * B + b) * DH + (size_t)d * H + j] + dh_rec[(size_t)b * H + j];
            if (cell == RNN_REF_LSTM) {
              double i = gt[j], f = gt[H + j], g = gt[2 * H + j], o = gt[3 * H + j];
              double c = R.c(st + 1, b)[j], cp = R.c(st, b)[j];
              double tau = std::tanh(c);
              double d_o = dh * tau;
              double dc = dc_rec[(size_t)b * H + j] + dh * o * (1.0 - tau * tau);
              double di = dc * g, dg = dc * i, df = dc * cp;
              dc_new[(size_t)b * H + j] = dc * f;
              gx[j] = di * i * (1.0 - i);
              gx[H + j] = df * f * (1.0 - f);
              gx[2 * H + j] = dg * (1.0 - g * g);
              gx[3 * H + j] = d_o * o * (1.0 - o);
              for (int q = 0; q < 4; ++q) gh[q * H + j] = gx[q * H + j];
              dh_new[(size_t)b * H + j] = 0.0;
            } else if (cell == RNN_REF_GRU) {
              double r = gt[j], z = gt[H + j], n = gt[2 * H + j];
              double hp = R.h(st, b)[j];
              double hn = R.n(st, b)[j];
              double dn = dh * (1.0 - z);
              double dz = dh * (hp - n);
              double dan = dn * (1.0 - n * n);
              double dr = dan * hn;
              double dhn = dan * r;
              gx[j] = dr * r * (1.0 - r);
              gx[H + j] = dz * z * (1.0 - z);
              gx[2 * H + j] = dan;
              gh[j] = gx[j];
              gh[H + j] = gx[H + j];
              gh[2 * H + j] = dhn;
              dh_new[(size_t)b * H + j] = dh * z;  // direct path h' = ... + z h
            } else if (cell == RNN_REF_RELU) {
              // d max(0, a)/da = 1 where the unit is on (a > 0), else 0
              gx[j] = R.o(st, b)[j] ? dh : 0.0;
              gh[j] = gx[j];
              dh_new[(size_t)b * H + j] = 0.0;
            } else {
              double h = gt[j];
              gx[j] = dh * (1.0 - h * h);
              gh[j] = gx[j];
              dh_new[(size_t)b * H + j] = 0.0;
            }
          }
        }
        // weight gradients of step st: dW_x += dGx^T in_t, dW_h += dGh^T h_prev
        if (dw) {
#pragma omp parallel for schedule(static)
          for (int p = 0; p < GH; ++p) {
            double* wxr = dW[v].Wx + (size_t)p * In;
            double* whr = dW[v].Wh + (size_t)p * H;
            double sbx = 0.0, sbh = 0.0;
            for (int b = 0; b < B; ++b) {
              const double* in = l == 0 ? x + ((size_t)t * B + b) * I : &out[l - 1][((size_t)t * B + b) * DH];
              const double* hp = R.h(st, b);
              double gxv = dGx[(size_t)b * GH + p], ghv = dGh[(size_t)b * GH + p];
              for (int k = 0; k < In; ++k) wxr[k] += gxv * in[k];
              for (int k = 0; k < H; ++k) whr[k] += ghv * hp[k];
              sbx += gxv;
              sbh += ghv;
            }
            dW[v].bx[p] += sbx;
            dW[v].bh[p] += sbh;
          }
        }
        // data gradients: d in_t += dGx W_x ; dh_prev = dGh W_h (+ direct term)
#pragma omp parallel for schedule(static)
        for (int b = 0; b < B; ++b) {
          double* din = &dbelow[((size_t)t * B + b) * In];
          double* dhp = &dh_new[(size_t)b * H];
          for (int p = 0; p < GH; ++p) {
            double gxv = dGx[(size_t)b * GH + p], ghv = dGh[(size_t)b * GH + p];
            const double* wxr = lw.Wx + (size_t)p * In;
            const double* whr = lw.Wh + (size_t)p * H;
            for (int k = 0; k < In; ++k) din[k] += gxv * wxr[k];
            for (int k = 0; k < H; ++k) dhp[k] += ghv * whr[k];
          }
        }
        dh_rec.swap(dh_new);
        if (cell == RNN_REF_LSTM) dc_rec.swap(dc_new);
      }
      if (dh0) std::memcpy(dh0 + (size_t)v * B * H, dh_rec.data(), sizeof(double) * B * H);
      if (dc0 && cell == RNN_REF_LSTM) std::memcpy(dc0 + (size_t)v * B * H, dc_rec.data(), sizeof(double) * B * H);
    }
    if (l == 0) {
      if (dx) std::memcpy(dx, dbelow.data(), sizeof(double) * (size_t)T * B * I);
    } else {
      dabove.swap(dbelow);
    }
  }
  return 0;
}

extern "C" int rnn_ref_bwd_dir(int cell, int L, int D, int T, int B, int I, int H, const int* lens,
                               const double* x, const double* h0, const double* c0, const double* w,
                               const double* dy, const double* dhT, const double* dcT, double* dx,
                               double* dh0, double* dc0, double* dw) {
  return rnn_ref_bwd_kp(cell, L, D, T, B, I, H, lens, 0, nullptr, x, h0, c0, w, dy, dhT, dcT, dx, dh0, dc0, dw);
}

extern "C" int rnn_ref_bwd_len(int cell, int L, int T, int B, int I, int H, const int* lens, const double* x,
                               const double* h0, const double* c0, const double* w,
                               const double* dy, const double* dhT, const double* dcT, double* dx,
                               double* dh0, double* dc0, double* dw) {
  return rnn_ref_bwd_dir(cell, L, 1, T, B, I, H, lens, x, h0, c0, w, dy, dhT, dcT, dx, dh0, dc0, dw);
}

extern "C" int rnn_ref_bwd(int cell, int L, int T, int B, int I, int H, const double* x,
                           const double* h0, const double* c0, const double* w,
                           const double* dy, const double* dhT, const double* dcT, double* dx,
                           double* dh0, double* dc0, double* dw) {
  return rnn_ref_bwd_dir(cell, L, 1, T, B, I, H, nullptr, x, h0, c0, w, dy, dhT, dcT, dx, dh0, dc0, dw);
}
