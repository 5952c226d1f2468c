// common.cuh -- types, conversions, error word and the cell arithmetic shared
// by every kernel of librnn.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace rnn {

enum Cell { LSTM = 0, GRU = 1, TANH = 2, RELU = 3 };

template <int CELL>
struct CellInfo;
template <>
struct CellInfo<LSTM> { static constexpr int G = 4; };
template <>
struct CellInfo<GRU> { static constexpr int G = 3; };
template <>
struct CellInfo<TANH> { static constexpr int G = 1; };
template <>
struct CellInfo<RELU> { static constexpr int G = 1; };

// Device error word codes (written into the first word of the workspace).
enum DevErr { DEV_OK = 0, DEV_TIMEOUT_PIPE = 1, DEV_TIMEOUT_STEP = 2, DEV_BAD_CLUSTER = 3 };

// ---------------------------------------------------------------- storage types
__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }
template <class S>
__device__ __forceinline__ S from_f32(float v);
template <>
__device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

// 16 consecutive elements of storage type S, to/from float.
template <class S>
__device__ __forceinline__ void load16(const S* p, float* v) {
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = to_f32(p[i]);
}
template <>
__device__ __forceinline__ void load16<float>(const float* p, float* v) {
  const float4* q = reinterpret_cast<const float4*>(p);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float4 f = q[i];
    v[4 * i] = f.x; v[4 * i + 1] = f.y; v[4 * i + 2] = f.z; v[4 * i + 3] = f.w;
  }
}
template <>
__device__ __forceinline__ void load16<__nv_bfloat16>(const __nv_bfloat16* p, float* v) {
  const uint4* q = reinterpret_cast<const uint4*>(p);
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    uint4 u = q[i];
    uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      v[8 * i + 2 * k] = __uint_as_float(w[k] << 16);
      v[8 * i + 2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
    }
  }
}
// 16 floats through L2 only (data written by other CTAs of the same launch).
__device__ __forceinline__ void load16_cg(const float* p, float* v) {
  const float4* q = reinterpret_cast<const float4*>(p);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float4 f = __ldcg(q + i);
    v[4 * i] = f.x; v[4 * i + 1] = f.y; v[4 * i + 2] = f.z; v[4 * i + 3] = f.w;
  }
}
template <class S>
__device__ __forceinline__ void store16(S* p, const float* v) {
#pragma unroll
  for (int i = 0; i < 16; ++i) p[i] = from_f32<S>(v[i]);
}
template <>
__device__ __forceinline__ void store16<float>(float* p, const float* v) {
  float4* q = reinterpret_cast<float4*>(p);
#pragma unroll
  for (int i = 0; i < 4; ++i) q[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
}
// One share of a 16-element store: elements e, e + es, ... (es a power of
// two; es = 1 is the whole vector store).
template <class S>
__device__ __forceinline__ void store16_share(S* p, const float* v, int e, int es) {
  if (es == 1) {
    store16(p, v);
    return;
  }
#pragma unroll
  for (int i = 0; i < 16; ++i)
    if ((i & (es - 1)) == e) p[i] = from_f32<S>(v[i]);
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}
template <>
__device__ __forceinline__ void store16<__nv_bfloat16>(__nv_bfloat16* p, const float* v) {
  uint4* q = reinterpret_cast<uint4*>(p);
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    q[i] = make_uint4(pack_bf16x2(v[8 * i], v[8 * i + 1]), pack_bf16x2(v[8 * i + 2], v[8 * i + 3]),
                      pack_bf16x2(v[8 * i + 4], v[8 * i + 5]), pack_bf16x2(v[8 * i + 6], v[8 * i + 7]));
  }
}

// ---------------------------------------------------------------- activations
// Precision of the pointwise cell arithmetic per storage type.  fp32 storage
// mode: every value the path stores is fp32 and the products run on FFMA, but
// the pointwise work between them (activations, cell update, the gate
// derivatives of the backward step) is evaluated in double from the stored
// fp32 inputs and rounded to fp32 once where it is stored, so each stored
// value carries a single fp32 rounding (CUDA's fp32 expf / tanhf and chains
// of fp32 operations carry several).  bf16 storage mode: fp32.
template <class S>
struct Prec {
  using T = double;
};
template <>
struct Prec<__nv_bfloat16> {
  using T = float;
};
// bf16 storage mode: the hardware tanh approximation (tanh.approx.f32, one
// special-function op, relative error about 2^-11) and the identity
// sigmoid(a) = (1 + tanh(a/2)) / 2.  The cell outputs are stored in bf16
// (relative step 2^-8), so the approximation stays below the storage rounding.
__device__ __forceinline__ float tanh_hw(float a) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(a));
  return y;
}
__device__ __forceinline__ float sigm_hw(float a) { return fmaf(0.5f, tanh_hw(0.5f * a), 0.5f); }
// activation pair for storage type S, in Prec<S>::T (fp32 storage: CUDA's
// double exp / tanh)
template <class S>
struct Act {
  __device__ __forceinline__ static double sig(double a) { return 1.0 / (1.0 + exp(-a)); }
  __device__ __forceinline__ static double th(double a) { return tanh(a); }
};
template <>
struct Act<__nv_bfloat16> {
  __device__ __forceinline__ static float sig(float a) { return sigm_hw(a); }
  __device__ __forceinline__ static float th(float a) { return tanh_hw(a); }
};

// Simple-RNN cells (one gate block): activation h = act(a) and its slope
// written in terms of h (tanh: 1 - h^2; ReLU: 1 where h > 0, taken as 0 at
// the kink).
template <int CELL, class S, class T>
__device__ __forceinline__ T simple_act(T a) {
  if constexpr (CELL == RELU) return a > T(0) ? a : T(0);
  else return Act<S>::th(a);
}
template <int CELL, class T>
__device__ __forceinline__ T simple_slope(T h) {
  if constexpr (CELL == RELU) return h > T(0) ? T(1) : T(0);
  else return T(1) - h * h;
}

// ---------------------------------------------------------------- time and errors
__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void raise_error(int* err, int code) {
  if (err) atomicCAS(err, 0, code);
}

// Packed gate-row index of (gate g, hidden unit j) with interleave block u:
// rows are grouped [H/u][G][u] so that one block of G*u rows holds every gate
// of u consecutive hidden units.
__device__ __forceinline__ int packed_row(int g, int j, int G, int u) {
  return (j / u) * (G * u) + g * u + (j % u);
}

}  // namespace rnn
