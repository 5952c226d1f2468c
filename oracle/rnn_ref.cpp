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
// The backward pass is the exact gradient of
//   L = sum(y*dy) + sum(hT*dhT) + sum(cT*dcT)
// taken in reverse time, top layer first, one step and one layer at a time
// (no reordering beyond the definition).
#include "rnn_ref.h"

#include <algorithm>
#include <cmath>
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

std::vector<LayerW> split_weights(const double* w, int G, int L, int I, int H) {
  std::vector<LayerW> v(L);
  const double* p = w;
  for (int l = 0; l < L; ++l) {
    int In = l == 0 ? I : H;
    v[l].In = In;
    v[l].Wx = p; p += (size_t)G * H * In;
    v[l].Wh = p; p += (size_t)G * H * H;
    v[l].bx = p; p += (size_t)G * H;
    v[l].bh = p; p += (size_t)G * H;
  }
  return v;
}

// Everything the backward pass needs from the forward pass, per layer.
struct Record {
  int T, B, H, G;
  std::vector<double> hs;     // (T+1) x B x H, slot 0 = h0, slot t+1 = h_t
  std::vector<double> cs;     // (T+1) x B x H (LSTM)
  std::vector<double> gates;  // T x B x G*H   activated gate values
  std::vector<double> hn;     // T x B x H     GRU: W_hn h_{t-1} + b_hn
  double* h(int t1, int b) { return &hs[((size_t)t1 * B + b) * H]; }
  double* c(int t1, int b) { return &cs[((size_t)t1 * B + b) * H]; }
  double* g(int t, int b) { return &gates[((size_t)t * B + b) * G * H]; }
  double* n(int t, int b) { return &hn[((size_t)t * B + b) * H]; }
};

bool bad_args(int cell, int L, int T, int B, int I, int H, const double* x, const double* w) {
  return cell < 0 || cell > 3 || L < 1 || T < 0 || B < 0 || I < 1 || H < 1 || (!x && T * B > 0) || !w;
}

// Forward over all layers; fills one Record per layer.
// lens (nullable = all T): sequence b runs steps 0 .. lens[b]-1; at later
// steps its state is carried unchanged (so slot T holds its final state) and
// its outputs are zero.
void forward(int cell, int L, int T, int B, int I, int H, const double* x, const double* h0,
             const double* c0, const std::vector<LayerW>& W, std::vector<Record>& rec, const int* lens) {
  const int G = gates_of(cell);
  const int GH = G * H;
  rec.assign(L, Record());
  for (int l = 0; l < L; ++l) {
    Record& R = rec[l];
    R.T = T; R.B = B; R.H = H; R.G = G;
    R.hs.assign((size_t)(T + 1) * B * H, 0.0);
    R.gates.assign((size_t)T * B * GH, 0.0);
    if (cell == RNN_REF_LSTM) R.cs.assign((size_t)(T + 1) * B * H, 0.0);
    if (cell == RNN_REF_GRU) R.hn.assign((size_t)T * B * H, 0.0);
    if (h0) std::memcpy(R.h(0, 0), h0 + (size_t)l * B * H, sizeof(double) * B * H);
    if (c0 && cell == RNN_REF_LSTM) std::memcpy(R.c(0, 0), c0 + (size_t)l * B * H, sizeof(double) * B * H);
    const LayerW& lw = W[l];
    std::vector<double> ax((size_t)B * GH), ah((size_t)B * GH);
    for (int t = 0; t < T; ++t) {
      // pre-activations: one dot product per (batch row, gate row)
#pragma omp parallel for collapse(2) schedule(static)
      for (int b = 0; b < B; ++b) {
        for (int p = 0; p < GH; ++p) {
          const double* in = l == 0 ? x + ((size_t)t * B + b) * I : rec[l - 1].h(t + 1, b);
          const double* hp = R.h(t, b);
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
          double* gt = R.g(t, b);
          double hprev = R.h(t, b)[j];
          double hnew;
          if (lens && t >= lens[b]) {
            // finished sequence: state carried, no gate values
            R.h(t + 1, b)[j] = hprev;
            if (cell == RNN_REF_LSTM) R.c(t + 1, b)[j] = R.c(t, b)[j];
            continue;
          }
          if (cell == RNN_REF_LSTM) {
            double i = sigm(sx[j] + sh[j]);
            double f = sigm(sx[H + j] + sh[H + j]);
            double g = std::tanh(sx[2 * H + j] + sh[2 * H + j]);
            double o = sigm(sx[3 * H + j] + sh[3 * H + j]);
            double c = f * R.c(t, b)[j] + i * g;
            hnew = o * std::tanh(c);
            R.c(t + 1, b)[j] = c;
            gt[j] = i; gt[H + j] = f; gt[2 * H + j] = g; gt[3 * H + j] = o;
          } else if (cell == RNN_REF_GRU) {
            double r = sigm(sx[j] + sh[j]);
            double z = sigm(sx[H + j] + sh[H + j]);
            double hn = sh[2 * H + j];
            double n = std::tanh(sx[2 * H + j] + r * hn);
            hnew = (1.0 - z) * n + z * hprev;
            R.n(t, b)[j] = hn;
            gt[j] = r; gt[H + j] = z; gt[2 * H + j] = n;
          } else if (cell == RNN_REF_RELU) {
            hnew = std::max(0.0, sx[j] + sh[j]);
            gt[j] = hnew;
          } else {
            hnew = std::tanh(sx[j] + sh[j]);
            gt[j] = hnew;
          }
          R.h(t + 1, b)[j] = hnew;
        }
      }
    }
  }
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

extern "C" int rnn_ref_fwd_len(int cell, int L, int T, int B, int I, int H, const int* lens, const double* x,
                               const double* h0, const double* c0, const double* w, double* y,
                               double* hT, double* cT) {
  if (bad_args(cell, L, T, B, I, H, x, w) || bad_lens(T, B, lens)) return -1;
  const int G = gates_of(cell);
  std::vector<LayerW> W = split_weights(w, G, L, I, H);
  std::vector<Record> rec;
  forward(cell, L, T, B, I, H, x, h0, c0, W, rec, lens);
  if (y && T > 0) {
    std::memcpy(y, rec[L - 1].h(1, 0), sizeof(double) * (size_t)T * B * H);
    if (lens)
      for (int t = 0; t < T; ++t)
        for (int b = 0; b < B; ++b)
          if (t >= lens[b]) std::memset(y + ((size_t)t * B + b) * H, 0, sizeof(double) * H);
  }
  for (int l = 0; l < L; ++l) {
    if (hT) std::memcpy(hT + (size_t)l * B * H, rec[l].h(T, 0), sizeof(double) * B * H);
    if (cT && cell == RNN_REF_LSTM)
      std::memcpy(cT + (size_t)l * B * H, rec[l].c(T, 0), sizeof(double) * B * H);
  }
  return 0;
}

extern "C" int rnn_ref_fwd(int cell, int L, int T, int B, int I, int H, const double* x,
                           const double* h0, const double* c0, const double* w, double* y,
                           double* hT, double* cT) {
  return rnn_ref_fwd_len(cell, L, T, B, I, H, nullptr, x, h0, c0, w, y, hT, cT);
}

extern "C" int rnn_ref_bwd_len(int cell, int L, int T, int B, int I, int H, const int* lens, const double* x,
                               const double* h0, const double* c0, const double* w,
                               const double* dy, const double* dhT, const double* dcT, double* dx,
                               double* dh0, double* dc0, double* dw) {
  if (bad_args(cell, L, T, B, I, H, x, w) || (!dy && T * B > 0) || bad_lens(T, B, lens)) return -1;
  const int G = gates_of(cell);
  const int GH = G * H;
  std::vector<LayerW> W = split_weights(w, G, L, I, H);
  std::vector<Record> rec;
  forward(cell, L, T, B, I, H, x, h0, c0, W, rec, lens);

  // gradient arriving at each layer's outputs h_t from above (dy for the top layer)
  std::vector<double> dabove(dy, dy + (size_t)T * B * H);
  // weight-gradient views into dw (same layout as w), zeroed first
  struct LayerDW { double *Wx, *Wh, *bx, *bh; };
  std::vector<LayerDW> dW(L);
  if (dw) {
    double* p = dw;
    for (int l = 0; l < L; ++l) {
      dW[l].Wx = p; p += (size_t)GH * W[l].In;
      dW[l].Wh = p; p += (size_t)GH * H;
      dW[l].bx = p; p += GH;
      dW[l].bh = p; p += GH;
    }
    std::memset(dw, 0, sizeof(double) * (size_t)(p - dw));
  }

  for (int l = L - 1; l >= 0; --l) {
    Record& R = rec[l];
    const LayerW& lw = W[l];
    const int In = lw.In;
    std::vector<double> dh_rec((size_t)B * H, 0.0), dc_rec((size_t)B * H, 0.0);
    if (dhT) std::memcpy(dh_rec.data(), dhT + (size_t)l * B * H, sizeof(double) * B * H);
    if (dcT && cell == RNN_REF_LSTM) std::memcpy(dc_rec.data(), dcT + (size_t)l * B * H, sizeof(double) * B * H);
    std::vector<double> dbelow((size_t)T * B * In, 0.0);  // gradient wrt this layer's inputs
    std::vector<double> dGx((size_t)B * GH), dGh((size_t)B * GH);
    std::vector<double> dh_new((size_t)B * H), dc_new((size_t)B * H);

    for (int t = T - 1; t >= 0; --t) {
      // pointwise: gate pre-activation gradients of step t
#pragma omp parallel for collapse(2) schedule(static)
      for (int b = 0; b < B; ++b) {
        for (int j = 0; j < H; ++j) {
          const double* gt = R.g(t, b);
          double* gx = &dGx[(size_t)b * GH];
          double* gh = &dGh[(size_t)b * GH];
          if (lens && t >= lens[b]) {
            // finished sequence: the step is the identity on the state and its
            // output is the constant 0, so the state gradient passes through
            for (int q = 0; q < G; ++q) gx[q * H + j] = gh[q * H + j] = 0.0;
            dh_new[(size_t)b * H + j] = dh_rec[(size_t)b * H + j];
            if (cell == RNN_REF_LSTM) dc_new[(size_t)b * H + j] = dc_rec[(size_t)b * H + j];
            continue;
          }
          double dh = dabove[((size_t)t * B + b) * H + j] + dh_rec[(size_t)b * H + j];
          if (cell == RNN_REF_LSTM) {
            double i = gt[j], f = gt[H + j], g = gt[2 * H + j], o = gt[3 * H + j];
            double c = R.c(t + 1, b)[j], cp = R.c(t, b)[j];
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
            double hp = R.h(t, b)[j];
            double hn = R.n(t, b)[j];
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
            // d max(0, a)/da = 1 where a > 0 (h > 0), else 0
            gx[j] = gt[j] > 0.0 ? dh : 0.0;
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
      // weight gradients of step t: dW_x += dGx^T in_t, dW_h += dGh^T h_{t-1}
      if (dw) {
#pragma omp parallel for schedule(static)
        for (int p = 0; p < GH; ++p) {
          double* wxr = dW[l].Wx + (size_t)p * In;
          double* whr = dW[l].Wh + (size_t)p * H;
          double sbx = 0.0, sbh = 0.0;
          for (int b = 0; b < B; ++b) {
            const double* in = l == 0 ? x + ((size_t)t * B + b) * I : rec[l - 1].h(t + 1, b);
            const double* hp = R.h(t, b);
            double gxv = dGx[(size_t)b * GH + p], ghv = dGh[(size_t)b * GH + p];
            for (int k = 0; k < In; ++k) wxr[k] += gxv * in[k];
            for (int k = 0; k < H; ++k) whr[k] += ghv * hp[k];
            sbx += gxv;
            sbh += ghv;
          }
          dW[l].bx[p] += sbx;
          dW[l].bh[p] += sbh;
        }
      }
      // data gradients: d in_t = dGx W_x ; dh_{t-1} = dGh W_h (+ direct term)
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
    if (dh0) std::memcpy(dh0 + (size_t)l * B * H, dh_rec.data(), sizeof(double) * B * H);
    if (dc0 && cell == RNN_REF_LSTM) std::memcpy(dc0 + (size_t)l * B * H, dc_rec.data(), sizeof(double) * B * H);
    if (l == 0) {
      if (dx) std::memcpy(dx, dbelow.data(), sizeof(double) * (size_t)T * B * I);
    } else {
      dabove.swap(dbelow);
    }
  }
  return 0;
}

extern "C" int rnn_ref_bwd(int cell, int L, int T, int B, int I, int H, const double* x,
                           const double* h0, const double* c0, const double* w,
                           const double* dy, const double* dhT, const double* dcT, double* dx,
                           double* dh0, double* dc0, double* dw) {
  return rnn_ref_bwd_len(cell, L, T, B, I, H, nullptr, x, h0, c0, w, dy, dhT, dcT, dx, dh0, dc0, dw);
}
