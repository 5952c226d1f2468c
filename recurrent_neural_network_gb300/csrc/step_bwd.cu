// step_bwd.cu -- one backward-through-time step of one layer: the product
// dGh_{s+1} W_h (gate gradients times the packed recurrent weights, read
// MN-major so that one packed copy serves both directions) with the pointwise
// gate derivative of step s fused into its epilogue; plus the pointwise-only
// first step of the reverse sweep.
//
// "Optimizing Performance of Recurrent Neural Networks on GPUs" (review page,
// section "제안 방법"): backward passes overlap across layers the same way as
// forward ones; the reverse sweep therefore has the same shape as the forward.
#include <cstring>

#include "epilogues.cuh"
#include "launch.cuh"

namespace rnn {

namespace {
template <int CELL, class S>
BwdPoint<CELL, S> make_point(const BwdStepArgs& a) {
  BwdPoint<CELL, S> p;
  p.B = a.B;
  p.H = a.H;
  p.u = a.u;
  p.gates = a.gates;
  p.c_s = a.c_s;
  p.c_sm1 = a.c_sm1;
  p.hn_s = a.hn_s;
  p.h_sm1 = static_cast<const S*>(a.h_sm1);
  p.dy = a.dy;
  p.dy_f32 = a.dy_f32;
  p.carry = a.carry;
  p.dGx = static_cast<S*>(a.dGx);
  p.dGh = static_cast<S*>(a.dGh);
  return p;
}

template <int CELL, class S>
EpiBwdStep<CELL, S> make_epi(const BwdStepArgs& a) {
  EpiBwdStep<CELL, S> e;
  e.pt = make_point<CELL, S>(a);
  e.final_ = a.final_;
  e.dh0 = static_cast<S*>(a.dh0);
  e.dc0 = a.dc0;
  e.part = a.part;
  e.counters = a.counters;
  e.err = nullptr;
  e.limit_ns = 0;
  return e;
}

template <int CELL>
int bwd_step_cell(const Launch& L, int mode, const Operand& A, const Operand& Bw, int bn, int splits,
                  const BwdStepArgs& a) {
  const int G = CellInfo<CELL>::G;
  const int M = a.B, N = a.H, K = G * a.H;
  if (mode == 1) {
    using S = __nv_bfloat16;
    auto e = make_epi<CELL, S>(a);
    e.err = L.err;
    e.limit_ns = L.limit_ns;
    // (CTA pairs inside split-K clusters measured slower here than 128-row
    // tiles in clusters of `splits`: 126 us vs 73 us per H=4096 B=256 step)
    if (bn == 256) return launch_tc<256, 4>(L, A, Bw, M, N, K, splits, 0, e, a.cluster_splitk != 0);
    if (bn == 128) return launch_tc<128, 6>(L, A, Bw, M, N, K, splits, 0, e, a.cluster_splitk != 0);
    return RNN_ERR_UNSUPPORTED;
  }
  return launch_simt<32>(L, A, Bw, M, N, K, make_epi<CELL, float>(a));
}

template <int CELL, class S>
__global__ void bwd_point_kernel(const BwdPoint<CELL, S> p, const S* __restrict__ dh_init) {
  const int chunks = p.H / 16;
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (long long)p.B * chunks) return;
  const int b = (int)(idx / chunks), j0 = (int)(idx % chunks) * 16;
  float dh[16];
  if (dh_init) load16(dh_init + (size_t)b * p.H + j0, dh);
  else
#pragma unroll
    for (int i = 0; i < 16; ++i) dh[i] = 0.f;
  p.run(b, j0, dh);
}

template <int CELL, class S>
int point_launch(const Launch& L, const BwdStepArgs& a, const void* dh_init) {
  const long long n = (long long)a.B * (a.H / 16);
  const int threads = 128;
  launch_begin(L);
  bwd_point_kernel<CELL, S><<<(unsigned)((n + threads - 1) / threads), threads, 0, L.stream>>>(
      make_point<CELL, S>(a), static_cast<const S*>(dh_init));
  cudaError_t e = cudaGetLastError();
  launch_end(L);
  return cuda_status(e);
}
}  // namespace

int bwd_step(const Launch& L, int mode, int cell, const Operand& A, const Operand& Bw, int bn, int splits,
             const BwdStepArgs& a) {
  if (cell == LSTM) return bwd_step_cell<LSTM>(L, mode, A, Bw, bn, splits, a);
  if (cell == GRU) return bwd_step_cell<GRU>(L, mode, A, Bw, bn, splits, a);
  if (cell == RELU) return bwd_step_cell<RELU>(L, mode, A, Bw, bn, splits, a);
  return bwd_step_cell<TANH>(L, mode, A, Bw, bn, splits, a);
}

int bwd_point(const Launch& L, int mode, int cell, const BwdStepArgs& a, const void* dh_init) {
  if (mode == 1) {
    using S = __nv_bfloat16;
    if (cell == LSTM) return point_launch<LSTM, S>(L, a, dh_init);
    if (cell == GRU) return point_launch<GRU, S>(L, a, dh_init);
    if (cell == RELU) return point_launch<RELU, S>(L, a, dh_init);
    return point_launch<TANH, S>(L, a, dh_init);
  }
  if (cell == LSTM) return point_launch<LSTM, float>(L, a, dh_init);
  if (cell == GRU) return point_launch<GRU, float>(L, a, dh_init);
  if (cell == RELU) return point_launch<RELU, float>(L, a, dh_init);
  return point_launch<TANH, float>(L, a, dh_init);
}

namespace {
template <int CELL>
__global__ void __launch_bounds__(256) bwd_point_v_kernel(const BwdPointV<CELL> p) {
  const long long q = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (q < (long long)p.B * (p.H / 4)) p.run(q);
}
}  // namespace


int bwd_dh_t(const Launch& L, const Operand& WhT, const Operand& dG, int B, int H, int G, int bn, int splits,
             float* dh, void* dh0, int final_, float* part, const float* pf_gates, const float* pf_c_s,
             const float* pf_c_sm1, const PointVArgs* fuse) {
  const int M = H, N = B, K = G * H;
  EpiBwdDhT e;
  std::memset(&e, 0, sizeof(e));
  e.B = B;
  e.H = H;
  e.dh = dh;
  e.dh0 = static_cast<__nv_bfloat16*>(dh0);
  e.final_ = final_;
  e.err = L.err;
  e.limit_ns = L.limit_ns;
  e.pf_gates = pf_gates;
  e.pf_c_s = pf_c_s;
  e.pf_c_sm1 = pf_c_sm1;
  e.G = G;
  // the K splits of a tile reduce inside a cluster (the only split-K path of
  // this epilogue): bn / splits must be a multiple of 16, at most 8 splits
  const int kb = (K + 63) / 64, sp = std::max(1, std::min(splits, kb));
  const int eff = (kb + (kb + sp - 1) / sp - 1) / ((kb + sp - 1) / sp);
  if (eff > 1 && (eff > 8 || bn % (16 * eff))) return RNN_ERR_UNSUPPORTED;
  // split partials meet in `part` ([eff][Bp][H], Bp = the batch rounded up
  // to whole tiles so that a tile's rows never spill into the next split)
  e.Bp = (B + bn - 1) / bn * bn;
  if (eff > 1) {
    if (!part) return RNN_ERR_INVALID_ARG;
    int rc = encode_plain(&e.map_part, part, 4, (long long)eff * e.Bp, H, H, 128, bn / eff);
    if (rc) return rc;
    if (!final_ && !fuse) {
      rc = encode_plain(&e.map_dh, dh, 4, B, H, H, 128, bn / eff);
      if (rc) return rc;
    }
  }
  if (fuse) {
    if (final_ || G != 4 || bn != 256 || eff != 4) return RNN_ERR_UNSUPPORTED;
    const PointVArgs& a = *fuse;
    int rc = encode_plain(&e.map_g, a.gates, 4, B, 4LL * H, 4LL * H, 256, 16);
    if (!rc) rc = encode_plain(&e.map_cs, a.c_s, 4, B, H, H, 128, 16);
    if (!rc && a.c_sm1) rc = encode_plain(&e.map_cp, a.c_sm1, 4, B, H, H, 128, 16);
    if (!rc) rc = encode_plain(&e.map_dc, a.carry, 4, B, H, H, 128, 16);
    if (!rc && a.dy) rc = encode_plain(&e.map_dy, a.dy, a.dy_f32 ? 4 : 2, B, H, H, 128, 16);
    if (rc) return rc;
    e.fuse = 1;
    e.has_cp = a.c_sm1 ? 1 : 0;
    e.has_dy = a.dy ? 1 : 0;
    e.dy_f32 = a.dy_f32;
    e.carry = a.carry;
    e.dc0 = a.dc0;
    e.dGx = static_cast<__nv_bfloat16*>(a.dGx);
  }
  if (bn == 256) return launch_tc<256, 4>(L, WhT, dG, M, N, K, splits, 0, e, true);
  if (bn == 128) return launch_tc<128, 6>(L, WhT, dG, M, N, K, splits, 0, e, true);
  if (bn == 64) return launch_tc<64, 8>(L, WhT, dG, M, N, K, splits, 0, e, true);
  return RNN_ERR_UNSUPPORTED;
}

int bwd_point_v(const Launch& L, int cell, const PointVArgs& a) {
  if (a.H % 4 || (cell != LSTM && cell != TANH && cell != RELU)) return RNN_ERR_UNSUPPORTED;
  const long long n = (long long)a.B * (a.H / 4);
  const int grid = (int)((n + 255) / 256);
  auto fill = [&](auto& p) {
    p.B = a.B;
    p.H = a.H;
    p.dh = a.dh;
    p.dh_init = static_cast<const __nv_bfloat16*>(a.dh_init);
    p.dy = a.dy;
    p.dy_f32 = a.dy_f32;
    p.gates = a.gates;
    p.c_s = a.c_s;
    p.c_sm1 = a.c_sm1;
    p.carry = a.carry;
    p.dc0 = a.dc0;
    p.dGx = static_cast<__nv_bfloat16*>(a.dGx);
  };
  launch_begin(L);
  if (cell == LSTM) {
    BwdPointV<LSTM> p;
    fill(p);
    bwd_point_v_kernel<LSTM><<<grid, 256, 0, L.stream>>>(p);
  } else {
    if (cell == RELU) {
      BwdPointV<RELU> p;
      fill(p);
      bwd_point_v_kernel<RELU><<<grid, 256, 0, L.stream>>>(p);
    } else {
      BwdPointV<TANH> p;
      fill(p);
      bwd_point_v_kernel<TANH><<<grid, 256, 0, L.stream>>>(p);
    }
  }
  const cudaError_t e = cudaGetLastError();
  launch_end(L);
  return cuda_status(e);
}

}  // namespace rnn
