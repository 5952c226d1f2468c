// stack.cuh -- pieces shared by the persistent stacked recurrences (forward
// in stack.cu, backward through time in stack_bwd.cu): the per-layer,
// per-timestep arrival counters, the asynchronous stores of the cross-chunk
// reduction inside a cluster, and the 3-D TMA maps that bring one CTA's
// whole K chunk of a timestep in one load.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>

#include "../../include/rnn.h"
#include "common.cuh"
#include "launch.cuh"
#include "tc.cuh"

namespace rnn {
namespace stk {

#define RNN_TRY_LOCAL(x)           \
  do {                             \
    const int rc_ = (x);           \
    if (rc_ != RNN_OK) return rc_; \
  } while (0)

__device__ __forceinline__ unsigned int ld_acquire_u32(const unsigned int* p) {
  unsigned int v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void red_release_add_u32(unsigned int* p, unsigned int v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// 16 bytes into the shared memory of a CTA of the cluster, counted (16
// transaction bytes) on that CTA's mbarrier
__device__ __forceinline__ void st_async_v4(uint32_t cluster_addr, const float* v, uint32_t cluster_bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
                   cluster_addr),
               "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
               "r"(__float_as_uint(v[3])), "r"(cluster_bar)
               : "memory");
}
__device__ __forceinline__ void st_dsmem_s32(uint32_t cluster_addr, int v) {
  asm volatile("st.shared::cluster.s32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}

// Raise the abort flag in every CTA of the cluster (this one included).
__device__ __forceinline__ void abort_cluster(volatile int* flag, int cluster) {
  *flag = 1;
  if (cluster > 1) {
    const uint32_t fa = tc::smem_addr(const_cast<int*>(flag));
    for (int r = 0; r < cluster; ++r) st_dsmem_s32(tc::mapa(fa, (uint32_t)r), 1);
  }
}

// Wait until *cnt >= want (bounded; gives up at once when the CTA aborts,
// and on timeout records DEV_TIMEOUT_STEP and aborts the cluster).
__device__ __forceinline__ bool wait_count(const unsigned int* cnt, unsigned int want, volatile int* abort_flag,
                                           int cluster, int* err, uint64_t limit_ns) {
  if (ld_acquire_u32(cnt) >= want) return true;
  const uint64_t t0 = globaltimer_ns();
  while (ld_acquire_u32(cnt) < want) {
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > limit_ns) {
      raise_error(err, DEV_TIMEOUT_STEP);
      abort_cluster(abort_flag, cluster);
      return false;
    }
  }
  return true;
}

// Bounded wait on an mbarrier whose bytes come from other CTAs of the
// cluster (acquire at cluster scope); gives up when the CTA aborts.
__device__ __forceinline__ bool wait_cluster_bytes(uint64_t* bar, uint32_t parity, volatile int* abort_flag, int* err,
                                                   uint64_t limit_ns) {
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (tc::mbar_try_wait_cluster(bar, parity)) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > limit_ns) {
      raise_error(err, DEV_TIMEOUT_STEP);
      return false;
    }
  }
}

// 3-D map over a sequence [rows][W] bf16 seen as (64 k, row, k block): box
// (64, N, nkb) with 128-byte swizzle; its shared-memory image is nkb
// consecutive N x 128-byte blocks, each one K-major tensor-core operand.
// Rows outside [0, rows) read zero.
inline int encode_seq3(CUtensorMap* map, const void* ptr, long long rows, int W, int N, int nkb) {
  auto enc = tmap_encoder();
  if (!enc) return RNN_ERR_CUDA;
  if ((reinterpret_cast<uintptr_t>(ptr) & 15) || W % 64) return RNN_ERR_INVALID_ARG;
  cuuint64_t dims[3] = {64, (cuuint64_t)rows, (cuuint64_t)(W / 64)};
  cuuint64_t strides[2] = {(cuuint64_t)W * 2, 128};
  cuuint32_t box[3] = {64, (cuuint32_t)N, (cuuint32_t)nkb}, es[3] = {1, 1, 1};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, es,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? RNN_OK : RNN_ERR_INVALID_ARG;
}

}  // namespace stk
}  // namespace rnn
