// gemm.cu -- the large products of the path (input projection over all
// timesteps, data gradient of the layer inputs, weight gradients over all
// timesteps), the weight pack and the bias-gradient reduction.
//
// "Optimizing Performance of Recurrent Neural Networks on GPUs" (review page,
// section "제안 방법"): the gate matrices are grouped into one larger product,
// the input product is independent of the recurrence, and the weight update
// is a single large product over all timesteps with a cheap bias update.
#include <algorithm>

#include <cuda_fp8.h>

#include "epilogues.cuh"
#include "launch.cuh"

namespace rnn {

namespace {
// BN choice for plain products: 256-wide tiles when N is large, 128 otherwise.
template <class OutT>
int run_store(const Launch& L, int mode, const Operand& A, const Operand& B, int M, int N, int K,
              const EpiStore<OutT>& epi, int max_ctas) {
  if (mode == 1) {
    if (N > 128 && M > 128 && L.pair) return launch_tc2<256, 6>(L, A, B, M, N, K, max_ctas, epi);
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

// ---------------------------------------------------------------- device copies and zero fills
// The copies and fills inside a call run as kernels on the SMs.  As
// copy-engine operations they would queue behind any large transfer the
// caller keeps running on a copy engine, e.g. the read-back of the previous
// step's weight gradients to the host, and hold the whole step up until it
// has finished.
namespace {
template <class V>
__global__ void copy2d_kernel(const uint8_t* __restrict__ src, size_t spitch, uint8_t* __restrict__ dst,
                              size_t dpitch, size_t w, size_t rows) {
  const size_t n = w * rows;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    const size_t r = rows == 1 ? 0 : i / w, c = rows == 1 ? i : i - r * w;
    reinterpret_cast<V*>(dst + r * dpitch)[c] = reinterpret_cast<const V*>(src + r * spitch)[c];
  }
}
template <class V>
__global__ void zero_kernel(V* __restrict__ dst, size_t n) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
    dst[i] = V{};
}
inline size_t align_of(uintptr_t v) { return v & 15 ? (v & 3 ? 1 : 4) : 16; }
int grid_for(const Launch& L, size_t n) { return (int)std::max<size_t>(1, std::min<size_t>((n + 255) / 256, (size_t)L.num_sms * 8)); }
}  // namespace

int dev_copy2d(const Launch& L, void* dst, size_t dpitch, const void* src, size_t spitch, size_t width, size_t rows) {
  if (!width || !rows) return RNN_OK;
  if (!dst || !src) return RNN_ERR_INVALID_ARG;
  const size_t a = std::min({align_of(reinterpret_cast<uintptr_t>(dst)), align_of(reinterpret_cast<uintptr_t>(src)),
                             align_of(rows > 1 ? dpitch : 16), align_of(rows > 1 ? spitch : 16), align_of(width)});
  const uint8_t* s = static_cast<const uint8_t*>(src);
  uint8_t* d = static_cast<uint8_t*>(dst);
  launch_begin(L);
  if (a == 16) {
    copy2d_kernel<uint4><<<grid_for(L, width / 16 * rows), 256, 0, L.stream>>>(s, spitch, d, dpitch, width / 16, rows);
  } else if (a == 4) {
    copy2d_kernel<uint32_t><<<grid_for(L, width / 4 * rows), 256, 0, L.stream>>>(s, spitch, d, dpitch, width / 4, rows);
  } else {
    copy2d_kernel<uint8_t><<<grid_for(L, width * rows), 256, 0, L.stream>>>(s, spitch, d, dpitch, width, rows);
  }
  const cudaError_t e = cudaGetLastError();
  launch_end(L);
  return cuda_status(e);
}

struct DevOps {
  DevOp op[kMaxDevOps];
};
namespace {
__global__ void batch_kernel(const __grid_constant__ DevOps ops) {
  const DevOp o = ops.op[blockIdx.y];
  const size_t stride = (size_t)gridDim.x * blockDim.x, i0 = blockIdx.x * (size_t)blockDim.x + threadIdx.x;
  const bool vec = !(reinterpret_cast<uintptr_t>(o.dst) & 15) && !(reinterpret_cast<uintptr_t>(o.src) & 15) &&
                   !(o.bytes & 15);
  if (vec) {
    uint4* d = static_cast<uint4*>(o.dst);
    const uint4* s = static_cast<const uint4*>(o.src);
    for (size_t i = i0; i < o.bytes / 16; i += stride) d[i] = s ? s[i] : make_uint4(0, 0, 0, 0);
  } else {
    uint8_t* d = static_cast<uint8_t*>(o.dst);
    const uint8_t* s = static_cast<const uint8_t*>(o.src);
    for (size_t i = i0; i < o.bytes; i += stride) d[i] = s ? s[i] : 0;
  }
}
}  // namespace

int dev_batch(const Launch& L, const DevOp* ops, int n) {
  for (int b = 0; b < n; b += kMaxDevOps) {
    DevOps p{};
    const int m = std::min(kMaxDevOps, n - b);
    size_t most = 0;
    for (int i = 0; i < m; ++i) {
      if (!ops[b + i].dst && ops[b + i].bytes) return RNN_ERR_INVALID_ARG;
      p.op[i] = ops[b + i];
      most = std::max(most, ops[b + i].bytes / 16 + (ops[b + i].bytes & 15));
    }
    if (!most) continue;
    launch_begin(L);
    batch_kernel<<<dim3(grid_for(L, most), m), 256, 0, L.stream>>>(p);
    const cudaError_t e = cudaGetLastError();
    launch_end(L);
    if (e != cudaSuccess) return cuda_status(e);
  }
  return RNN_OK;
}

int dev_copy(const Launch& L, void* dst, const void* src, size_t bytes) {
  return dev_copy2d(L, dst, bytes, src, bytes, bytes, 1);
}

int dev_zero(const Launch& L, void* dst, size_t bytes) {
  if (!bytes) return RNN_OK;
  if (!dst) return RNN_ERR_INVALID_ARG;
  const size_t a = std::min(align_of(reinterpret_cast<uintptr_t>(dst)), align_of(bytes));
  launch_begin(L);
  if (a == 16) zero_kernel<uint4><<<grid_for(L, bytes / 16), 256, 0, L.stream>>>(static_cast<uint4*>(dst), bytes / 16);
  else if (a == 4) zero_kernel<uint32_t><<<grid_for(L, bytes / 4), 256, 0, L.stream>>>(static_cast<uint32_t*>(dst), bytes / 4);
  else zero_kernel<uint8_t><<<grid_for(L, bytes), 256, 0, L.stream>>>(static_cast<uint8_t*>(dst), bytes);
  const cudaError_t e = cudaGetLastError();
  launch_end(L);
  return cuda_status(e);
}

// ---------------------------------------------------------------- f32 -> bf16 copy
__global__ void cast_bf16_kernel(const float4* __restrict__ src, uint2* __restrict__ dst, size_t n4) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n4; i += (size_t)gridDim.x * blockDim.x) {
    const float4 v = src[i];
    const __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
    dst[i] = make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&b));
  }
}

int cast_bf16(const Launch& L, const float* src, void* dst, size_t n) {
  if (n % 4 || (reinterpret_cast<uintptr_t>(src) & 15) || (reinterpret_cast<uintptr_t>(dst) & 15))
    return RNN_ERR_INVALID_ARG;
  const size_t n4 = n / 4;
  if (n4 == 0) return RNN_OK;
  const int blocks = (int)std::min<size_t>((n4 + 255) / 256, (size_t)L.num_sms * 8);
  launch_begin(L);
  cast_bf16_kernel<<<blocks, 256, 0, L.stream>>>(reinterpret_cast<const float4*>(src), static_cast<uint2*>(dst), n4);
  cudaError_t e = cudaGetLastError();
  launch_end(L);
  return cuda_status(e);
}

// ---------------------------------------------------------------- fp8 stash of W_h
// One block per row: the row's largest magnitude, the scale that maps it to
// the largest finite e4m3 value (448), and every element divided by the scale
// and rounded to the nearest e4m3 value (ties to even; CUDA's conversion).
__global__ void quant_rows_kernel(const __nv_bfloat16* __restrict__ w, int cols, uint8_t* __restrict__ q,
                                  float* __restrict__ scale) {
  __shared__ float red[32];
  const __nv_bfloat16* row = w + (size_t)blockIdx.x * cols;
  float m = 0.f;
  for (int k = threadIdx.x; k < cols; k += blockDim.x) m = fmaxf(m, fabsf(__bfloat162float(row[k])));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  m = 0.f;
  for (int i = 0; i < (int)(blockDim.x >> 5); ++i) m = fmaxf(m, red[i]);
  const float s = m > 0.f ? m / 448.f : 1.f;
  if (threadIdx.x == 0) scale[blockIdx.x] = s;
  uint8_t* qr = q + (size_t)blockIdx.x * cols;
  for (int k = threadIdx.x; k < cols; k += blockDim.x)
    qr[k] = (uint8_t)__nv_cvt_float_to_fp8(__bfloat162float(row[k]) / s, __NV_SATFINITE, __NV_E4M3);
}

int quant_rows_e4m3(const Launch& L, const void* w, int rows, int cols, uint8_t* q, float* scale) {
  if (rows <= 0 || cols <= 0 || !w || !q || !scale) return RNN_ERR_INVALID_ARG;
  launch_begin(L);
  quant_rows_kernel<<<rows, 256, 0, L.stream>>>(static_cast<const __nv_bfloat16*>(w), cols, q, scale);
  cudaError_t e = cudaGetLastError();
  launch_end(L);
  return cuda_status(e);
}

// ---------------------------------------------------------------- bias gradient
// db[user col] = sum over rows of dG[row][packed col].  Pass 1: each block
// owns 256 packed columns (32 lanes x 8 columns, 16-byte loads) and one slice
// of rows, its 8 warps stride the slice and reduce through shared memory into
// a per-slice partial.  Pass 2 sums the slices in a fixed order, so the result
// is deterministic.  In the fp32 storage mode both passes sum with
// compensation (TwoSum, as in the fp32 GEMM engine), so that the bias
// gradients carry about one rounding error whatever the number of rows.
template <class S>
__global__ void bias_part_kernel(const S* __restrict__ dg, float* __restrict__ part, long long rows, int GH,
                                 long long rows_per_slice) {
  __shared__ float red[8][256];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c0 = blockIdx.x * 256 + lane * 8;
  const long long r0 = (long long)blockIdx.y * rows_per_slice;
  const long long r1 = min(rows, r0 + rows_per_slice);
  constexpr bool comp = sizeof(S) == 4;
  float acc[8], err[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = err[i] = 0.f;
  if (c0 < GH) {
    for (long long r = r0 + warp; r < r1; r += 8) {
      const S* p = dg + r * GH + c0;
      if (sizeof(S) == 2) {
        uint4 u = *reinterpret_cast<const uint4*>(p);
        uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          acc[2 * k] += __uint_as_float(w[k] << 16);
          acc[2 * k + 1] += __uint_as_float(w[k] & 0xFFFF0000u);
        }
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) sum2_add(to_f32(p[i]), acc[i], err[i]);
      }
    }
  }
  __shared__ float rerr[comp ? 8 : 1][comp ? 256 : 1];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    red[warp][lane * 8 + i] = acc[i];
    if constexpr (comp) rerr[warp][lane * 8 + i] = err[i];
  }
  __syncthreads();
  const int c = threadIdx.x;  // 256 threads: one column each
  float t = 0.f, te = 0.f;
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    if constexpr (comp) {
      sum2_add(red[w][c], t, te);
      te = __fadd_rn(te, rerr[w][c]);
    } else {
      t += red[w][c];
    }
  }
  const int col = blockIdx.x * 256 + c;
  if (col < GH) part[(size_t)blockIdx.y * GH + col] = comp ? __fadd_rn(t, te) : t;
}

__global__ void bias_final_kernel(const float* __restrict__ part, int slices, int G, int H, int u,
                                  float* __restrict__ db, float* __restrict__ db2, int accumulate) {
  const int p = blockIdx.x * blockDim.x + threadIdx.x;
  const int GH = G * H;
  if (p >= GH) return;
  float t = 0.f, te = 0.f;  // compensated: costs nothing next to the loads
  for (int s = 0; s < slices; ++s) sum2_add(part[(size_t)s * GH + p], t, te);
  t = __fadd_rn(t, te);
  const int blk = p / (G * u), r = p % (G * u);
  const int ur = (r / u) * H + blk * u + (r % u);
  db[ur] = accumulate ? db[ur] + t : t;
  if (db2) db2[ur] = accumulate ? db2[ur] + t : t;  // same column sums, second destination
}

int bias_grad(const Launch& L, int mode, int cell, int H, int u, long long rows, const void* dgx, const void* dgh,
              float* dbx, float* dbh, int accumulate, float* part, int slices) {
  const int G = cell == LSTM ? 4 : cell == GRU ? 3 : 1;
  const int GH = G * H;
  if (GH % 8 || slices < 1) return RNN_ERR_INVALID_ARG;
  const long long per = (rows + slices - 1) / slices;
  dim3 grid((GH + 255) / 256, slices);
  // LSTM and RNN share one gate-gradient matrix between the input and the
  // recurrent side: reduce it once and write both bias gradients
  const int passes = dgx == dgh ? 1 : 2;
  launch_begin(L);
  for (int which = 0; which < passes; ++which) {
    const void* dg = which == 0 ? dgx : dgh;
    float* db = which == 0 ? dbx : dbh;
    float* db2 = passes == 1 ? dbh : nullptr;
    if (mode == 1)
      bias_part_kernel<__nv_bfloat16><<<grid, 256, 0, L.stream>>>(static_cast<const __nv_bfloat16*>(dg), part, rows,
                                                                  GH, per);
    else
      bias_part_kernel<float><<<grid, 256, 0, L.stream>>>(static_cast<const float*>(dg), part, rows, GH, per);
    bias_final_kernel<<<(GH + 255) / 256, 256, 0, L.stream>>>(part, slices, G, H, u, db, db2, accumulate);
  }
  cudaError_t e = cudaGetLastError();
  launch_end(L, 2 * passes);
  return cuda_status(e);
}

}  // namespace rnn
