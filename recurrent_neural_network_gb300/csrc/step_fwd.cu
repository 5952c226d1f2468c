// step_fwd.cu -- one forward timestep of one layer: the recurrent product
// h_{t-1} W_h^T on the tensor cores (bf16) or FFMA (fp32) with the gate
// non-linearities and the cell/state update fused into its epilogue.
//
// "Optimizing Performance of Recurrent Neural Networks on GPUs" (review page,
// section "제안 방법"): grouped gate matrices make each step one larger
// product; "Persistent RNNs: Stashing Recurrent Weights On-Chip" (citing
// snippets on its page) counts the pointwise work as cheap next to the
// products, which is why it runs inside the product's epilogue.
#include <cstring>

#include "epilogues.cuh"
#include "launch.cuh"

namespace rnn {

namespace {
template <int CELL, class S>
EpiFwdStep<CELL, S> make_epi(const FwdStepArgs& a) {
  EpiFwdStep<CELL, S> e;
  e.B = a.B;
  e.H = a.H;
  e.u = a.u;
  e.P = a.P;
  e.write_gates = a.write_gates;
  e.bias_hn = a.bias_hn;
  e.c_prev = a.c_prev;
  e.c_out = a.c_out;
  e.h_prev = static_cast<const S*>(a.h_prev);
  e.h_out = static_cast<S*>(a.h_out);
  e.y = static_cast<S*>(a.y);
  e.hT = static_cast<S*>(a.hT);
  e.cT = a.cT;
  e.hn_out = a.hn_out;
  return e;
}
}  // namespace

int fwd_step(const Launch& L, int mode, int cell, const Operand& A, const Operand& Bw, const FwdStepArgs& a) {
  const int G = cell == LSTM ? 4 : cell == GRU ? 3 : 1;
  const int M = a.B, N = G * a.H, K = a.H;
  if (mode == 1) {
    using S = __nv_bfloat16;
    // the tile width is one packed block of G*u gate rows
    // more than 128 batch rows: 256-row tiles on CTA pairs
    if (M > 128 && L.pair) {
      if (cell == LSTM && a.u == 64) return launch_tc2<256, 6>(L, A, Bw, M, N, K, 0, make_epi<LSTM, S>(a));
      if (cell == LSTM && a.u == 32) return launch_tc2<128, 8>(L, A, Bw, M, N, K, 0, make_epi<LSTM, S>(a));
      if (cell == LSTM && a.u == 16) return launch_tc2<64, 10>(L, A, Bw, M, N, K, 0, make_epi<LSTM, S>(a));
      if (cell == GRU && a.u == 64) return launch_tc2<192, 7>(L, A, Bw, M, N, K, 0, make_epi<GRU, S>(a));
      if (cell == GRU && a.u == 32) return launch_tc2<96, 9>(L, A, Bw, M, N, K, 0, make_epi<GRU, S>(a));
      if (cell == TANH && a.u == 128) return launch_tc2<128, 8>(L, A, Bw, M, N, K, 0, make_epi<TANH, S>(a));
      if (cell == RELU && a.u == 128) return launch_tc2<128, 8>(L, A, Bw, M, N, K, 0, make_epi<RELU, S>(a));
    }
#define RNN_STEP(C, U, BN_, ST)     \
  if (cell == C && a.u == U) return launch_tc<BN_, ST>(L, A, Bw, M, N, K, 1, 0, make_epi<C, S>(a));
    RNN_STEP(LSTM, 64, 256, 4) RNN_STEP(LSTM, 32, 128, 6) RNN_STEP(LSTM, 16, 64, 8)
    RNN_STEP(GRU, 64, 192, 5) RNN_STEP(GRU, 32, 96, 7) RNN_STEP(GRU, 16, 48, 8)
    RNN_STEP(TANH, 128, 128, 6) RNN_STEP(TANH, 64, 64, 8) RNN_STEP(TANH, 32, 32, 8)
    RNN_STEP(RELU, 128, 128, 6) RNN_STEP(RELU, 64, 64, 8) RNN_STEP(RELU, 32, 32, 8)
#undef RNN_STEP
    return RNN_ERR_UNSUPPORTED;
  }
  using S = float;
  if (cell == LSTM && a.u == 32) return launch_simt<128>(L, A, Bw, M, N, K, make_epi<LSTM, S>(a));
  if (cell == GRU && a.u == 32) return launch_simt<96>(L, A, Bw, M, N, K, make_epi<GRU, S>(a));
  if (cell == TANH && a.u == 32) return launch_simt<32>(L, A, Bw, M, N, K, make_epi<TANH, S>(a));
  if (cell == RELU && a.u == 32) return launch_simt<32>(L, A, Bw, M, N, K, make_epi<RELU, S>(a));
  return RNN_ERR_UNSUPPORTED;
}

namespace {
template <int CELL>
EpiFwdStepT<CELL> make_epi_t(const FwdStepArgs& a, int bn) {
  using S = __nv_bfloat16;
  EpiFwdStepT<CELL> e;
  std::memset(&e, 0, sizeof(e));
  e.B = a.B;
  e.H = a.H;
  e.P = a.P;
  e.write_gates = a.write_gates;
  e.c_prev = a.c_prev;
  e.c_out = a.c_out;
  e.h_out = static_cast<S*>(a.h_out);
  e.y = static_cast<S*>(a.y);
  e.hT = static_cast<S*>(a.hT);
  e.cT = a.cT;
  // several steps in one launch: the sequences' rows of all of them
  const int steps = a.steps > 1 ? a.steps : 1, rs = a.B * steps;
  e.step_rows = a.B;
  e.hT_step = steps > 1 ? a.hT_step : 0;
  e.step_cnt = steps > 1 ? a.step_cnt : nullptr;
  // bulk-store maps for the single-tile path; any failure keeps plain stores
  const int G = CellInfo<CELL>::G, ku = EpiFwdStepT<CELL>::kUnits;
  constexpr int rows = 32;  // batch rows per bulk store
  (void)bn;
  int rc = encode_plain(&e.map_p, a.P, 4, rs, (long long)G * a.H, (long long)G * a.H, 128, rows);
  if (!rc && CELL == LSTM) rc = encode_plain(&e.map_c, a.c_out, 4, rs, a.H, a.H, ku, rows);
  if (!rc && CELL == LSTM && a.cT) rc = encode_plain(&e.map_cT, a.cT, 4, a.B, a.H, a.H, ku, rows);
  if (!rc) rc = encode_plain(&e.map_h, a.h_out, 2, rs, a.H, a.H, ku, rows);
  if (!rc && a.y) rc = encode_plain(&e.map_y, a.y, 2, rs, a.H, a.H, ku, rows);
  if (!rc && a.hT) rc = encode_plain(&e.map_hT, a.hT, 2, a.B, a.H, a.H, ku, rows);
  e.tma_out = rc == RNN_OK ? 1 : 0;
  return e;
}

// the shared-SM variant: the same fields, every map with 16-row boxes
int make_epi_tr(const Launch& L, const FwdStepArgs& a, EpiFwdStepTR<LSTM>* e) {
  std::memset(e, 0, sizeof(*e));
  static_cast<EpiFwdStepT<LSTM>&>(*e) = make_epi_t<LSTM>(a, 256);
  constexpr int rows = EpiFwdStepTR<LSTM>::kRows, ku = EpiFwdStepTR<LSTM>::kU;
  int rc = encode_plain(&e->map_p, a.P, 4, a.B, 4LL * a.H, 4LL * a.H, 128, rows);
  if (!rc) rc = encode_plain(&e->map_c, a.c_out, 4, a.B, a.H, a.H, ku, rows);
  if (!rc && a.cT) rc = encode_plain(&e->map_cT, a.cT, 4, a.B, a.H, a.H, ku, rows);
  if (!rc) rc = encode_plain(&e->map_h, a.h_out, 2, a.B, a.H, a.H, ku, rows);
  if (!rc && a.y) rc = encode_plain(&e->map_y, a.y, 2, a.B, a.H, a.H, ku, rows);
  if (!rc && a.hT) rc = encode_plain(&e->map_hT, a.hT, 2, a.B, a.H, a.H, ku, rows);
  e->err = L.err;
  e->limit_ns = L.limit_ns;
  return rc;
}
}  // namespace

int fwd_step_t(const Launch& L, int cell, const Operand& Wh, const Operand& Hp, const FwdStepArgs& a) {
  const int G = cell == LSTM ? 4 : (cell == TANH || cell == RELU) ? 1 : 0;
  if (!G || a.u != 1) return RNN_ERR_UNSUPPORTED;
  const int M = G * a.H, N = a.B, K = a.H;
  if (a.steps > 1) {
    // the LSTM steps of a chunk in one cooperative launch: a pair loads h of
    // step s-1 once all pairs have stored it (each pair's two CTAs arrive
    // once per half of their epilogue warps); the bulk stores of 32 batch rows
    // must not reach into the next step's rows
    if (cell != LSTM || a.slim || !a.step_cnt || N % 32) return RNN_ERR_UNSUPPORTED;
    Operand Hs = Hp;
    Hs.mn_ext = N * a.steps;
    const int bn = N > 128 ? 256 : N > 64 ? 128 : 64;
    const EpiFwdStepT<LSTM> e = make_epi_t<LSTM>(a, bn);
    if (!e.tma_out) return RNN_ERR_UNSUPPORTED;
    if (bn == 256) return launch_tc2<256, 6>(L, Wh, Hs, M, N, K, 0, e, 1, a.steps, N, a.step_cnt, 4);
    if (bn == 128) return launch_tc2<128, 8>(L, Wh, Hs, M, N, K, 0, e, 1, a.steps, N, a.step_cnt, 4);
    return launch_tc2<64, 10>(L, Wh, Hs, M, N, K, 0, e, 1, a.steps, N, a.step_cnt, 4);
  }
  // one n-tile holds the whole batch (up to 256 entries): W_h streams once per step
#define RNN_STEP_T(BN_, ST)                                                                          \
  if (cell == LSTM) return launch_tc2<BN_, ST>(L, Wh, Hp, M, N, K, 0, make_epi_t<LSTM>(a, BN_));      \
  if (cell == RELU) return launch_tc2<BN_, ST>(L, Wh, Hp, M, N, K, 0, make_epi_t<RELU>(a, BN_));      \
  return launch_tc2<BN_, ST>(L, Wh, Hp, M, N, K, 0, make_epi_t<TANH>(a, BN_));
  if (N > 128 && cell == LSTM && a.slim) {
    // three stages and one accumulator: 97.5 KB of shared memory and 256 TMEM
    // columns, so that a CTA of another launch (the next layer's step) fits
    // beside each of these
    static_assert(tce2::smem_bytes<256, 3>() + 1024 <= (227 * 1024) / 2, "two CTAs per SM");
    static_assert(2 * EpiFwdStepTR<LSTM>::kPartBytes <= 3 * tce2::stage_bytes<256>(), "slots in the stages");
    EpiFwdStepTR<LSTM> e;
    const int rc = make_epi_tr(L, a, &e);
    if (rc) return rc;
    return launch_tc2<256, 3, EpiFwdStepTR<LSTM>, 1>(L, Wh, Hp, M, N, K, 0, e);
  }
  if (N > 128) {
    RNN_STEP_T(256, 6)
  }
  if (N > 64) {
    RNN_STEP_T(128, 8)
  }
  RNN_STEP_T(64, 10)
#undef RNN_STEP_T
}

}  // namespace rnn
