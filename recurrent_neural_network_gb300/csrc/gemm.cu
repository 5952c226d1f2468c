// gemm.cu -- the large products of the path (input projection over all
// timesteps, data gradient of the layer inputs, weight gradients over all
// timesteps), the weight pack and the bias-gradient reduction.
//
// "Optimizing Performance of Recurrent Neural Networks on GPUs" (review page,
// section "제안 방법"): the gate matrices are grouped into one larger product,
// the input product is independent of the recurrence, and the weight update
// is a single large product over all timesteps with a cheap bias update.
#include "epilogues.cuh"
#include "launch.cuh"

namespace rnn {

namespace {
// BN choice for plain products: 256-wide tiles when N is large, 128 otherwise.
template <class OutT>
int run_store(const Launch& L, int mode, const Operand& A, const Operand& B, int M, int N, int K,
              const EpiStore<OutT>& epi, int max_ctas) {
  if (mode == 1) {
    if (N > 128) return launch_tc<256, 4>(L, A, B, M, N, K, 1, max_ctas, epi);
    return launch_tc<128, 6>(L, A, B, M, N, K, 1, max_ctas, epi);
  }
  return launch_simt<64>(L, A, B, M, N, K, epi);
}
}  // namespace

int gemm_f32(const Launch& L, int mode, const Operand& A, const Operand& B, int M, int N, int K, float* D,
             long long ldd, const float* bias, int accumulate, const Remap& remap, int max_ctas) {
  EpiStore<float> e{D, ldd, M, N, bias, accumulate, remap.on, remap.G, remap.u, remap.H};
  return run_store(L, mode, A, B, M, N, K, e, max_ctas);
}

int gemm_store(const Launch& L, int mode, const Operand& A, const Operand& B, int M, int N, int K, void* D,
               long long ldd, int max_ctas) {
  if (mode == 1) {
    EpiStore<__nv_bfloat16> e{static_cast<__nv_bfloat16*>(D), ldd, M, N, nullptr, 0, 0, 1, 1, 1};
    return run_store(L, mode, A, B, M, N, K, e, max_ctas);
  }
  EpiStore<float> e{static_cast<float*>(D), ldd, M, N, nullptr, 0, 0, 1, 1, 1};
  return run_store(L, mode, A, B, M, N, K, e, max_ctas);
}

// ---------------------------------------------------------------- weight pack
template <class S>
__global__ void pack_rows_kernel(const S* __restrict__ w, S* __restrict__ pw, int G, int H, int K, int u) {
  // one block-row per packed row p; user row = g*H + j
  const int p = blockIdx.x;
  const int blk = p / (G * u), r = p % (G * u);
  const int g = r / u, j = blk * u + (r % u);
  const S* src = w + (size_t)(g * H + j) * K;
  S* dst = pw + (size_t)p * K;
  for (int k = threadIdx.x; k < K; k += blockDim.x) dst[k] = src[k];
}

template <class S>
__global__ void pack_bias_kernel(const S* __restrict__ bx, const S* __restrict__ bh, float* __restrict__ pb,
                                 float* __restrict__ pbn, int cell, int G, int H, int u) {
  const int p = blockIdx.x * blockDim.x + threadIdx.x;
  if (p >= G * H) return;
  const int blk = p / (G * u), r = p % (G * u);
  const int g = r / u, j = blk * u + (r % u);
  const int ur = g * H + j;
  const float x = to_f32(bx[ur]), h = to_f32(bh[ur]);
  // LSTM / RNN fold both biases into the input projection; GRU keeps b_hn
  // apart because the reset gate multiplies it.
  if (cell == GRU && g == 2) {
    pb[p] = x;
    pbn[j] = h;
  } else {
    pb[p] = x + h;
  }
}

int pack_layer(const Launch& L, int mode, int cell, int H, int In, int u, const void* wx, const void* wh,
               const void* bx, const void* bh, void* pwx, void* pwh, float* pbias, float* pbias_hn) {
  const int G = cell == LSTM ? 4 : cell == GRU ? 3 : 1;
  const int GH = G * H;
  launch_begin(L);
  if (mode == 1) {
    using S = __nv_bfloat16;
    pack_rows_kernel<S><<<GH, 128, 0, L.stream>>>(static_cast<const S*>(wx), static_cast<S*>(pwx), G, H, In, u);
    pack_rows_kernel<S><<<GH, 128, 0, L.stream>>>(static_cast<const S*>(wh), static_cast<S*>(pwh), G, H, H, u);
    pack_bias_kernel<S><<<(GH + 255) / 256, 256, 0, L.stream>>>(static_cast<const S*>(bx), static_cast<const S*>(bh),
                                                                pbias, pbias_hn, cell, G, H, u);
  } else {
    using S = float;
    pack_rows_kernel<S><<<GH, 128, 0, L.stream>>>(static_cast<const S*>(wx), static_cast<S*>(pwx), G, H, In, u);
    pack_rows_kernel<S><<<GH, 128, 0, L.stream>>>(static_cast<const S*>(wh), static_cast<S*>(pwh), G, H, H, u);
    pack_bias_kernel<S><<<(GH + 255) / 256, 256, 0, L.stream>>>(static_cast<const S*>(bx), static_cast<const S*>(bh),
                                                                pbias, pbias_hn, cell, G, H, u);
  }
  cudaError_t e = cudaGetLastError();
  launch_end(L, 3);
  return cuda_status(e);
}

// ---------------------------------------------------------------- bias gradient
// db[user col] = sum over rows of dG[row][packed col]; 32 packed columns per
// block, 8 row groups reduced through shared memory.
template <class S>
__global__ void bias_grad_kernel(const S* __restrict__ dgx, const S* __restrict__ dgh, float* __restrict__ dbx,
                                 float* __restrict__ dbh, long long rows, int G, int H, int u, int accumulate) {
  __shared__ float sx[8][33], sh[8][33];
  const int GH = G * H;
  const int p = blockIdx.x * 32 + threadIdx.x;
  float ax = 0.f, ah = 0.f;
  if (p < GH) {
    for (long long r = threadIdx.y; r < rows; r += 8) {
      ax += to_f32(dgx[r * GH + p]);
      ah += to_f32(dgh[r * GH + p]);
    }
  }
  sx[threadIdx.y][threadIdx.x] = ax;
  sh[threadIdx.y][threadIdx.x] = ah;
  __syncthreads();
  if (threadIdx.y == 0 && p < GH) {
    float tx = 0.f, th = 0.f;
    for (int i = 0; i < 8; ++i) {
      tx += sx[i][threadIdx.x];
      th += sh[i][threadIdx.x];
    }
    const int blk = p / (G * u), r = p % (G * u);
    const int ur = (r / u) * H + blk * u + (r % u);
    if (accumulate) {
      dbx[ur] += tx;
      dbh[ur] += th;
    } else {
      dbx[ur] = tx;
      dbh[ur] = th;
    }
  }
}

int bias_grad(const Launch& L, int mode, int cell, int H, int u, long long rows, const void* dgx, const void* dgh,
              float* dbx, float* dbh, int accumulate) {
  const int G = cell == LSTM ? 4 : cell == GRU ? 3 : 1;
  dim3 grid((G * H + 31) / 32), block(32, 8);
  launch_begin(L);
  if (mode == 1) {
    using S = __nv_bfloat16;
    bias_grad_kernel<S><<<grid, block, 0, L.stream>>>(static_cast<const S*>(dgx), static_cast<const S*>(dgh), dbx,
                                                      dbh, rows, G, H, u, accumulate);
  } else {
    using S = float;
    bias_grad_kernel<S><<<grid, block, 0, L.stream>>>(static_cast<const S*>(dgx), static_cast<const S*>(dgh), dbx,
                                                      dbh, rows, G, H, u, accumulate);
  }
  cudaError_t e = cudaGetLastError();
  launch_end(L);
  return cuda_status(e);
}

}  // namespace rnn
